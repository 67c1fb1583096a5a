// simt_gemm.cu -- FP32 SIMT GEMM (exact class): C = A * B, row-major fp32.
//
// The register-tiled shared-memory kernel of "Optimizing a WebGPU Matmul
// Kernel using Subgroups" (section 4 shared-memory tiles, section 5 a block of
// outputs per thread, section 6 unrolled loops, section 7 128-bit loads and
// stores), sized for an sm_103a SM instead of the page's 8 x 8 workgroup:
//
//   * a CTA of 256 threads computes a 128 x 128 tile of C; each thread owns
//     an 8 x 8 register tile laid out as 2 x 2 blocks of 4 x 4 (rows ty*4 and
//     64 + ty*4, columns tx*4 and 64 + tx*4) so that every shared-memory
//     fragment read is one 128-bit load shared by many lanes (a broadcast);
//   * K advances in slices of 8; A is staged transposed (k-major, padded to
//     132 floats per k-row so the transposing stores do not conflict) and B
//     as is; two shared-memory buffers and a register prefetch overlap the
//     global loads of slice s + 1 with the FMAs of slice s;
//   * global loads and stores are 128-bit and coalesced when the operands
//     allow (VEC), otherwise scalar; both forms zero-fill outside the
//     matrices and guard every store, the boundary rule of section 4 of
//     "WebGPU WGSL Compute Shaders: Custom Matrix Multiplication (GEMM)
//     Optimization Guide".
//
// Each output is accumulated by fused multiply-adds over k in increasing
// order in fp32, so |C - AB| <= K 2^-24 |A||B| element-wise.

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gemm {
namespace {

constexpr int kTile = 128;
constexpr int kSliceK = 8;
constexpr int kThreads = 256;
constexpr int kApad = kTile + 4;
constexpr int kGroup = 8;  // raster group height in tiles (L2 reuse)

struct SimtParams {
  int M, N, K;
  const float *A;
  long long lda;
  const float *B;
  long long ldb;
  float *C;
  long long ldc;
  int tiles_m, tiles_n;
};

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2) simt_gemm_kernel(const SimtParams p) {
  __shared__ __align__(16) float As[2][kSliceK][kApad];
  __shared__ __align__(16) float Bs[2][kSliceK][kTile];

  // Grouped raster: kGroup tile-rows sweep all tile-columns before moving on.
  const int bid = blockIdx.x;
  const int group_tiles = kGroup * p.tiles_n;
  const int g = bid / group_tiles;
  const int first_m = g * kGroup;
  const int gm_cnt = min(p.tiles_m - first_m, kGroup);
  const int r = bid - g * group_tiles;
  const int m0 = (first_m + r % gm_cnt) * kTile;
  const int n0 = (r / gm_cnt) * kTile;

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;

  // Load assignment: A row (tid / 2), k-offset (tid % 2) * 4;
  // B k-row (tid / 32), column (tid % 32) * 4.
  const int a_row = tid >> 1, a_k = (tid & 1) * 4;
  const int b_k = tid >> 5, b_col = (tid & 31) * 4;
  const int ga_row = m0 + a_row;
  const int gb_col = n0 + b_col;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  float a_reg[4], b_reg[4];

  auto load_slice = [&](int k0) {
    const int ka = k0 + a_k;
    const int kb = k0 + b_k;
    if (VEC) {
      // K % 4 == 0 and N % 4 == 0: a 4-wide group is wholly inside or outside.
      float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
      if (ga_row < p.M && ka < p.K)
        va = __ldg(reinterpret_cast<const float4 *>(p.A + static_cast<long long>(ga_row) * p.lda + ka));
      if (kb < p.K && gb_col < p.N)
        vb = __ldg(reinterpret_cast<const float4 *>(p.B + static_cast<long long>(kb) * p.ldb + gb_col));
      a_reg[0] = va.x; a_reg[1] = va.y; a_reg[2] = va.z; a_reg[3] = va.w;
      b_reg[0] = vb.x; b_reg[1] = vb.y; b_reg[2] = vb.z; b_reg[3] = vb.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a_reg[j] = (ga_row < p.M && ka + j < p.K)
                       ? __ldg(p.A + static_cast<long long>(ga_row) * p.lda + ka + j)
                       : 0.0f;
        b_reg[j] = (kb < p.K && gb_col + j < p.N)
                       ? __ldg(p.B + static_cast<long long>(kb) * p.ldb + gb_col + j)
                       : 0.0f;
      }
    }
  };
  auto store_slice = [&](int buf) {
#pragma unroll
    for (int j = 0; j < 4; ++j) As[buf][a_k + j][a_row] = a_reg[j];
    *reinterpret_cast<float4 *>(&Bs[buf][b_k][b_col]) =
        make_float4(b_reg[0], b_reg[1], b_reg[2], b_reg[3]);
  };

  const int num_slices = (p.K + kSliceK - 1) / kSliceK;
  load_slice(0);
  store_slice(0);
  __syncthreads();

  for (int s = 0; s < num_slices; ++s) {
    const int buf = s & 1;
    const bool more = s + 1 < num_slices;
    if (more) load_slice((s + 1) * kSliceK);
#pragma unroll
    for (int k = 0; k < kSliceK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][k][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][k][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][k][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][k][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) store_slice(buf ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (row >= p.M) continue;
    float *crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = n0 + h * 64 + tx * 4;
      if (VEC) {
        if (col < p.N)
          *reinterpret_cast<float4 *>(crow + col) =
              make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (col + j < p.N) crow[col + j] = acc[i][h * 4 + j];
      }
    }
  }
}

}  // namespace

int simt_launch(const GemmArgs &a, cudaStream_t stream) {
  SimtParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.A = a.A;
  p.lda = a.lda;
  p.B = a.B;
  p.ldb = a.ldb;
  p.C = a.C;
  p.ldc = a.ldc;
  p.tiles_m = static_cast<int>((a.M + kTile - 1) / kTile);
  p.tiles_n = static_cast<int>((a.N + kTile - 1) / kTile);
  const long long blocks = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (blocks > 0x7fffffffLL) return kErrInvalidArg;
  const bool vec = reinterpret_cast<uintptr_t>(a.A) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.B) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.lda % 4 == 0 &&
                   a.ldb % 4 == 0 && a.ldc % 4 == 0 && a.K % 4 == 0 && a.N % 4 == 0;
  if (vec)
    simt_gemm_kernel<true><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
  else
    simt_gemm_kernel<false><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace gemm
