// checks.cuh -- device-side index checks of the checked build.
//
// The library is also built as libgemm_f32_checked.so, from the same sources
// with GEMM_F32_INDEX_CHECKS=1. In that build every global-memory access that
// a kernel addresses with its own index arithmetic is first compared with the
// extent, in elements, that the host declared for the buffer: plain loads of
// A and B, stores (and beta reads) of C, the stream-K and cluster-split
// partial slots and counters, the shared-memory band of a cluster-split sum,
// the operand copies and the reduction. An access whose offset range
// [offset, offset + len) is not inside [0, extent) is skipped -- the kernel
// goes on, no fault and no trap -- and the first such access of each
// translation unit is recorded, with a count of all of them, in that unit's
// IndexFault record; gemm_f32_take_index_fault reads and clears the records.
// TMA copies need no check here: the tensor map's extents bound them in
// hardware (a box past an edge is zero-filled, never read from outside).
//
// In the regular build (GEMM_F32_INDEX_CHECKS undefined or 0) index_ok is
// the constant true and every check compiles away.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#ifndef GEMM_F32_INDEX_CHECKS
#define GEMM_F32_INDEX_CHECKS 0
#endif

namespace gemm {

// First recorded violation of a translation unit and the number of them.
struct IndexFault {
  unsigned count;
  int site;
  long long offset;
  long long extent;
};

// Where an access was checked (values of gemm_f32_take_index_fault's site).
enum IndexSite : int {
  kSiteNone = 0,
  kSiteCStore = 1,         // C element stored (or read for beta) by a kernel's epilogue
  kSitePartialWrite = 2,   // stream-K / cluster-split partial slot written
  kSitePartialRead = 3,    // partial slot read by a split-tile or cluster-split sum
  kSiteCounter = 4,        // split-tile arrival counter
  kSiteBand = 5,           // cluster-split band in shared memory
  kSiteLoadA = 6,          // plain load (or asynchronous copy) of A
  kSiteLoadB = 7,          // plain load (or asynchronous copy) of B
  kSiteCopySrc = 8,        // operand copy / transpose: source read
  kSiteCopyDst = 9,        // operand copy / transpose: destination written
  kSiteReduceIn = 10,      // reduction input read
  kSiteReducePartial = 11, // reduction partial written or read
  kSiteReduceOut = 12,     // reduction result written
  kSiteCount
};

#if GEMM_F32_INDEX_CHECKS
namespace {

// This translation unit's record (each unit of the library is its own device
// module).
__device__ IndexFault g_index_fault;

__device__ __noinline__ void index_fault_record(int site, long long offset, long long extent) {
  if (atomicAdd(&g_index_fault.count, 1u) == 0u) {
    g_index_fault.site = site;
    g_index_fault.offset = offset;
    g_index_fault.extent = extent;
  }
}

}  // namespace
#endif

// True if elements [offset, offset + len) of a buffer of `extent` elements may
// be accessed. In the checked build a false result records the violation and
// the caller skips the access.
__device__ __forceinline__ bool index_ok(int site, long long offset, long long len,
                                         long long extent) {
#if GEMM_F32_INDEX_CHECKS
  if (offset >= 0 && offset + len <= extent) return true;
  index_fault_record(site, offset, extent);
  return false;
#else
  (void)site;
  (void)offset;
  (void)len;
  (void)extent;
  return true;
#endif
}

// The same for a pointer into a buffer that starts at `base`.
__device__ __forceinline__ bool ptr_ok(int site, const void *ptr, long long len,
                                       const float *base, long long extent) {
#if GEMM_F32_INDEX_CHECKS
  return index_ok(site, static_cast<const float *>(ptr) - base, len, extent);
#else
  (void)site;
  (void)ptr;
  (void)len;
  (void)base;
  (void)extent;
  return true;
#endif
}

// Extent in elements of a rows x cols matrix with row pitch ld (0 if empty).
__host__ __device__ constexpr long long matrix_extent(long long rows, long long cols,
                                                      long long ld) {
  return rows > 0 && cols > 0 ? (rows - 1) * ld + cols : 0;
}

}  // namespace gemm

// Defines `int NAME(IndexFault *out, bool clear)` on the host: copy this
// translation unit's record to *out and, with clear, reset it (the caller has
// synchronised). In the regular build the record does not exist and *out is
// zeroed without a device access.
#if GEMM_F32_INDEX_CHECKS
#define GEMM_INDEX_FAULT_TAKE(NAME)                                                        \
  int NAME(IndexFault *out, bool clear) {                                                  \
    const IndexFault zero = {0u, 0, 0, 0};                                                 \
    if (cudaMemcpyFromSymbol(out, g_index_fault, sizeof(IndexFault)) != cudaSuccess)       \
      return kErrLaunch;                                                                   \
    if (clear && out->count != 0u &&                                                       \
        cudaMemcpyToSymbol(g_index_fault, &zero, sizeof(IndexFault)) != cudaSuccess)       \
      return kErrLaunch;                                                                   \
    return kOk;                                                                            \
  }
#else
#define GEMM_INDEX_FAULT_TAKE(NAME)           \
  int NAME(IndexFault *out, bool /*clear*/) { \
    *out = IndexFault{0u, 0, 0, 0};           \
    return kOk;                               \
  }
#endif
