// kernels.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units. Internal to libgemm_f32.so.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "checks.cuh"

namespace gemm {

// C = alpha * op(A) op(B) + beta * C, row-major. opa = 0: A is M x K (pitch
// lda); opa = 1: A is stored transposed, K x M. opb = 0: B is K x N (pitch
// ldb); opb = 1: B is stored transposed, N x K.
struct GemmArgs {
  int64_t M, N, K;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
  int opb = 0;
  int opa = 0;
  float alpha = 1.0f;
  float beta = 0.0f;
  // Extent of C in elements that the kernels' index checks hold stores to
  // (checked build); -1: the extent of the M x N matrix, (M - 1) ldc + N.
  int64_t c_extent = -1;
};

// The extent index checks use for C.
inline long long c_extent_of(const GemmArgs &a) {
  return a.c_extent >= 0 ? a.c_extent : matrix_extent(a.M, a.N, a.ldc);
}

// Status codes (values of gemm_f32_status).
enum : int {
  kOk = 0,
  kErrInvalidArg = 1,
  kErrUnsupportedDevice = 2,
  kErrLaunch = 3,
  kErrTimeout = 4,
  kErrAlias = 5,
  kErrIndex = 6,
};

// True when A and B as given can be described by TMA tensor maps: A not
// stored transposed, 16-byte aligned base addresses and row pitches that are
// multiples of 16 bytes.
bool tc_tma_direct(const GemmArgs &a);

// tcgen05 GEMM: exact = 3xTF32, else single-pass TF32; lsu = operands staged
// by plain loads instead of TMA. The TMA-fed kernel takes any operands: those
// that are not tc_tma_direct are first copied (A stored transposed:
// transposed) into a workspace from the library's pool that is. Requires
// K >= 1, M >= 1, N >= 1.
int tc_launch(const GemmArgs &a, bool exact, bool lsu, int sm_count, cudaStream_t stream);

// Words of a streamed launch, in device memory (see TcParams::stream_*).
// Rows of A and of C go in groups of `group` rows of unit tiles
// (kStreamRows rows of the matrices each): a_ready[i] = epoch once group i's
// rows of A have landed; b_ready[0] = epoch once B's rows [0, 32 kb_split)
// have, and b_ready[1] once the rest have; c_done[i] counts the CTAs that
// stored their part of a unit tile of group i of C (zeroed before the
// launch; the group is complete at tc_stream_done_target(N, its rows of unit
// tiles)).
struct StreamFeed {
  const unsigned *a_ready = nullptr;
  const unsigned *b_ready = nullptr;
  unsigned *c_done = nullptr;
  unsigned epoch = 0;
  int kb_split = 0;
  int group = 1;
  // Limit of each device-side wait, 0 for the kernel's default (self-test).
  unsigned long long timeout_ns = 0;
};
constexpr int kStreamRows = 256;     // rows of A and of C per row of unit tiles
// Value to which a streamed launch that gives up (and the host, should it
// ever have to) raises the done counters. The return stream's waits compare
// cyclically, (int32_t)(counter - target) >= 0, so the value must stay at
// least every target (below 2^27) and far from 2^31 when late increments
// add to it: 2^30.
constexpr unsigned kStreamRelease = 0x40000000u;
constexpr int kStreamKBlock = 32;    // k per k-block of kb_split
inline unsigned tc_stream_done_target(int64_t N, int64_t tile_rows) {
  // two CTAs per 256-column unit tile
  return static_cast<unsigned>(2 * ((N + 255) / 256) * tile_rows);
}

// One persistent launch of the TMA-fed 3xTF32 pair kernel over whole unit
// tiles in row-major order, its producers waiting on feed's words before
// copying operands and its epilogue counting the stored tiles per group. A
// (M x K) and B (K x N), not stored transposed, must be tc_tma_direct; K >= 1.
int tc_launch_streamed(const GemmArgs &a, const StreamFeed &feed, int sm_count,
                       cudaStream_t stream);

// tc_launch with the stream-K workspace in the library's fixed scratch array
// (no allocation, so no operand copies: with lsu = false the operands must
// be tc_tma_direct). Returns kErrInvalidArg if the problem needs more scratch
// than GEMM_F32_NOALLOC_SCRATCH_BYTES.
int tc_launch_noalloc(const GemmArgs &a, bool exact, bool lsu, int sm_count, cudaStream_t stream);

// dst (cols x rows, pitch ldd) = src^T for src rows x cols (pitch lds), on
// `stream`. Sizes below 2^31.
int transpose_launch(const float *src, int64_t lds, int64_t rows, int64_t cols, float *dst,
                     int64_t ldd, int sm_count, cudaStream_t stream);

// Stream-ordered workspace from the library's memory pool on the current
// device (kept reserved by the pool once used, never shrunk).
int pool_alloc(void **ptr, size_t bytes, cudaStream_t stream);
int pool_free(void *ptr, cudaStream_t stream);

// Sum of x[0, n) into *out (device pointers): `groups` partial sums written to
// `partials` (groups floats), then a second kernel adds them. n == 0 sets
// *out = 0.
int reduce_launch(int64_t n, const float *x, float *out, int groups, float *partials,
                  cudaStream_t stream);
int reduce_default_groups(int sm_count);

// One row-by-row copy: dst (rows x cols, pitch ldd) = src (pitch lds). Sizes
// below 2^31 columns; rows <= 0 or cols <= 0 is an empty job.
struct PackJob {
  const float *src = nullptr;
  int64_t lds = 0, rows = 0, cols = 0;
  float *dst = nullptr;
  int64_t ldd = 0;
  // Declared extents (elements) of src and dst for the index checks; set by
  // pack_rows_launch from the shape.
  int64_t src_extent = 0, dst_extent = 0;
};

// Both jobs in one launch on `stream`.
int pack_rows_launch(const PackJob &first, const PackJob &second, int sm_count,
                     cudaStream_t stream);

// Rates of the TF32 tensor pipe (MMA-only kernel) and of the FP32 FMA pipe
// (FFMA-only kernel) on sm_count SMs, in TFLOP/s, and the median SM clock
// (MHz) each kernel's CTAs ran at. Blocking.
int probe_peaks(int sm_count, double *tf32_tflops, double *fp32_tflops, double *tf32_mhz,
                double *fp32_mhz, cudaStream_t stream);

// SIMT FP32 GEMM. Requires M >= 1, N >= 1 (K = 0 stores beta * C).
// may_alloc: A stored M x K may first be transposed into a workspace from
// the library's pool (see simt_gemm.cu); false where nothing may be
// allocated (gemm_f32_noalloc).
int simt_launch(const GemmArgs &a, int sm_count, bool may_alloc, cudaStream_t stream);

// Synchronise `stream`, then read and clear the device status word.
int tc_poll_status(cudaStream_t stream);

// Bounded-wait self-test (see gemm_f32_selftest_wait_timeout).
int tc_selftest_wait_timeout(int64_t timeout_ns, cudaStream_t stream);

// Abort-path self-test (see gemm_f32_selftest_stalled_gemm): the TMA-fed pair
// kernel of the mode with its producers stopping after one k-block; returns
// the device status read after the launch.
int tc_selftest_stalled_gemm(const GemmArgs &a, bool exact, int64_t timeout_ns, int sm_count,
                             cudaStream_t stream);

// Checked build: read (and with clear, reset) the index-check record of
// each translation unit (see checks.cuh); the caller has synchronised the
// device. In the regular build they return an empty record.
int tc_index_fault_take(IndexFault *out, bool clear);
int simt_index_fault_take(IndexFault *out, bool clear);
int pack_index_fault_take(IndexFault *out, bool clear);
int transpose_index_fault_take(IndexFault *out, bool clear);
int reduce_index_fault_take(IndexFault *out, bool clear);

}  // namespace gemm
