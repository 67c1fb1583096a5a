// pack.cu -- strided fp32 matrix copy into a 16-byte row pitch.
//
// TMA tensor maps need 16-byte aligned bases and row pitches that are
// multiples of 16 bytes. An operand outside that rule (an odd leading
// dimension, or a base offset by 4, 8 or 12 bytes) is copied once into a
// library workspace that meets it, and the TMA-fed tensor-core kernel reads
// the copy: a copy bound by HBM bandwidth instead of a GEMM whose operand
// tiles must be gathered with plain loads.
//
// A CTA of 256 threads copies whole rows, the rows taken in steps of the grid;
// each warp reads and writes 128 consecutive bytes per instruction (one
// coalesced segment), four instructions in flight per thread. Both operands
// of a GEMM that need it are copied by one launch.

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gemm {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

// Copies the rows of up to two matrices in one launch (a GEMM's operands are
// copied together: one launch less ahead of the GEMM). Rows [0, first.rows)
// of the combined row range belong to `first`, the rest to `second`.
__global__ void __launch_bounds__(kThreads)
    pack_rows_kernel(const PackJob first, const PackJob second) {
  // The GEMM that reads the copies is launched as a programmatic dependent:
  // let it start its set-up now (it waits for this grid before reading).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long total = first.rows + second.rows;
  for (long long rr = blockIdx.x; rr < total; rr += gridDim.x) {
    const bool in_first = rr < first.rows;
    const PackJob &j = in_first ? first : second;
    const long long r = in_first ? rr : rr - first.rows;
    const float *s = j.src + r * j.lds;
    float *d = j.dst + r * j.ldd;
    const int cols = static_cast<int>(j.cols);
    // Index checks of the checked build (checks.cuh); nothing in the regular one.
    auto load = [&](int cc) {
      return index_ok(kSiteCopySrc, r * j.lds + cc, 1, j.src_extent) ? __ldg(s + cc) : 0.0f;
    };
    auto store = [&](int cc, float v) {
      if (index_ok(kSiteCopyDst, r * j.ldd + cc, 1, j.dst_extent)) d[cc] = v;
    };
    int c = threadIdx.x;
    for (; c + 3 * kThreads < cols; c += 4 * kThreads) {
      const float v0 = load(c), v1 = load(c + kThreads), v2 = load(c + 2 * kThreads),
                  v3 = load(c + 3 * kThreads);
      store(c, v0);
      store(c + kThreads, v1);
      store(c + 2 * kThreads, v2);
      store(c + 3 * kThreads, v3);
    }
    for (; c < cols; c += kThreads) store(c, load(c));
  }
}

}  // namespace

GEMM_INDEX_FAULT_TAKE(pack_index_fault_take)

int pack_rows_launch(const PackJob &first, const PackJob &second, int sm_count,
                     cudaStream_t stream) {
  const long long total = (first.rows > 0 && first.cols > 0 ? first.rows : 0) +
                          (second.rows > 0 && second.cols > 0 ? second.rows : 0);
  if (total <= 0) return kOk;
  PackJob a = first, b = second;
  if (a.rows <= 0 || a.cols <= 0) a.rows = 0;
  if (b.rows <= 0 || b.cols <= 0) b.rows = 0;
  for (PackJob *j : {&a, &b}) {
    j->src_extent = matrix_extent(j->rows, j->cols, j->lds);
    j->dst_extent = matrix_extent(j->rows, j->cols, j->ldd);
  }
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * kBlocksPerSm;
  const unsigned grid = static_cast<unsigned>(total < cap ? total : cap);
  pack_rows_kernel<<<grid, kThreads, 0, stream>>>(a, b);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace gemm
