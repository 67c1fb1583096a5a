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
// coalesced segment), four instructions in flight per thread.

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gemm {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

__global__ void __launch_bounds__(kThreads)
    pack_rows_kernel(const float *__restrict__ src, long long lds, int rows, int cols,
                     float *__restrict__ dst, long long ldd) {
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const float *s = src + static_cast<long long>(r) * lds;
    float *d = dst + static_cast<long long>(r) * ldd;
    int c = threadIdx.x;
    for (; c + 3 * kThreads < cols; c += 4 * kThreads) {
      const float v0 = __ldg(s + c), v1 = __ldg(s + c + kThreads), v2 = __ldg(s + c + 2 * kThreads),
                  v3 = __ldg(s + c + 3 * kThreads);
      d[c] = v0;
      d[c + kThreads] = v1;
      d[c + 2 * kThreads] = v2;
      d[c + 3 * kThreads] = v3;
    }
    for (; c < cols; c += kThreads) d[c] = __ldg(s + c);
  }
}

}  // namespace

int pack_rows_launch(const float *src, int64_t lds, int64_t rows, int64_t cols, float *dst,
                     int64_t ldd, int sm_count, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return kOk;
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * kBlocksPerSm;
  const unsigned grid = static_cast<unsigned>(rows < cap ? rows : cap);
  pack_rows_kernel<<<grid, kThreads, 0, stream>>>(src, lds, static_cast<int>(rows),
                                                  static_cast<int>(cols), dst, ldd);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace gemm
