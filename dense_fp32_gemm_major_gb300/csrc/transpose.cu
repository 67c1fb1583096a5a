// transpose.cu -- out-of-place fp32 matrix transpose, dst = src^T.
//
// Feeds the TMA-fed tensor-core kernel when A is supplied transposed (stored
// K x M): TMA can only hand the tcgen05 TF32 MMA K-major tiles, so A^T is
// first rewritten as a row-major M x K copy with a 16-byte pitch. The copy is
// bound by HBM bandwidth (one read and one write of the matrix).
//
// A CTA of 256 threads moves 64 x 64 tiles through shared memory (a padded
// 64 x 65 array, so that the column reads of the transposed store do not
// conflict): loads and stores are each one coalesced 128-byte row segment
// per warp, sixteen loads in flight per thread (the copy is bound by how many
// bytes are in flight per SM). CTAs are persistent and walk the tiles in
// steps of the grid.

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gemm {
namespace {

constexpr int kT = 64;            // tile edge
constexpr int kW = 32;            // columns per warp access
constexpr int kRowsPerPass = 8;   // 256 threads = 8 warps
constexpr int kBlocksPerSm = 32;  // grid cap: up to one tile per CTA at the usual sizes

__global__ void __launch_bounds__(kW * kRowsPerPass)
    transpose_kernel(const float *__restrict__ src, long long lds, int rows, int cols,
                     float *__restrict__ dst, long long ldd, int tiles_c, long long tiles,
                     long long src_extent, long long dst_extent) {
  __shared__ float t[kT][kT + 1];
  // The GEMM that reads the copy is launched as a programmatic dependent:
  // let it start its set-up now (it waits for this grid before reading).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tx = threadIdx.x % kW, ty = threadIdx.x / kW;
  for (long long tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int r0 = static_cast<int>(tile / tiles_c) * kT;
    const int c0 = static_cast<int>(tile % tiles_c) * kT;
    float v[kT / kRowsPerPass][2];
#pragma unroll
    for (int i = 0; i < kT / kRowsPerPass; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = r0 + ty + i * kRowsPerPass, c = c0 + tx + h * kW;
        const long long off = static_cast<long long>(r) * lds + c;
        v[i][h] = (r < rows && c < cols && index_ok(kSiteCopySrc, off, 1, src_extent))
                      ? __ldg(src + off)
                      : 0.0f;
      }
#pragma unroll
    for (int i = 0; i < kT / kRowsPerPass; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) t[ty + i * kRowsPerPass][tx + h * kW] = v[i][h];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kT / kRowsPerPass; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = c0 + ty + i * kRowsPerPass, r = r0 + tx + h * kW;  // dst row c, column r
        const long long off = static_cast<long long>(c) * ldd + r;
        if (c < cols && r < rows && index_ok(kSiteCopyDst, off, 1, dst_extent))
          dst[off] = t[tx + h * kW][ty + i * kRowsPerPass];
      }
    __syncthreads();
  }
}

}  // namespace

GEMM_INDEX_FAULT_TAKE(transpose_index_fault_take)

int transpose_launch(const float *src, int64_t lds, int64_t rows, int64_t cols, float *dst,
                     int64_t ldd, int sm_count, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return kOk;
  const long long tiles_r = (rows + kT - 1) / kT, tiles_c = (cols + kT - 1) / kT;
  const long long tiles = tiles_r * tiles_c;
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * kBlocksPerSm;
  const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
  transpose_kernel<<<grid, kW * kRowsPerPass, 0, stream>>>(
      src, lds, static_cast<int>(rows), static_cast<int>(cols), dst, ldd,
      static_cast<int>(tiles_c), tiles, matrix_extent(rows, cols, lds),
      matrix_extent(cols, rows, ldd));
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace gemm
