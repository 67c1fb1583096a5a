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
// order in fp32, so |C - AB| <= K 2^-24 |A||B| element-wise. The general form
// C = alpha * A op(B) + beta * C scales the sum once at the store (C is read
// only when beta != 0). op(B) = B, or B stored transposed (N x K, the vec4
// transposed-B storage of the subgroups page, section 7), which is staged
// through the same transposing stores as A; op(A) = A, or A stored
// transposed (K x M), whose rows of m are stored into the k-major tile as is.

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
  float alpha, beta;
  int tiles_m, tiles_n;
};

template <bool VEC, bool OPB, bool OPA>
__global__ void __launch_bounds__(kThreads, 2) simt_gemm_kernel(const SimtParams p) {
  __shared__ __align__(16) float As[2][kSliceK][kApad];
  __shared__ __align__(16) float Bs[2][kSliceK][kApad];

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

  // Load assignment: A row (tid / 2), k-offset (tid % 2) * 4 (A stored
  // transposed: k-row tid / 32, rows (tid % 32) * 4 ...); B k-row (tid / 32),
  // column (tid % 32) * 4, or for B stored transposed, like A: n-row
  // (tid / 2), k-offset (tid % 2) * 4.
  const int a_row = OPA ? (tid & 31) * 4 : tid >> 1;
  const int a_k = OPA ? tid >> 5 : (tid & 1) * 4;
  const int b_k = OPB ? (tid & 1) * 4 : tid >> 5;
  const int b_col = OPB ? tid >> 1 : (tid & 31) * 4;
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
      // Contiguous extents are multiples of 4: a 4-wide group is wholly
      // inside or outside.
      float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
      if (OPA) {
        if (ka < p.K && ga_row < p.M)
          va = __ldg(reinterpret_cast<const float4 *>(p.A + static_cast<long long>(ka) * p.lda + ga_row));
      } else if (ga_row < p.M && ka < p.K) {
        va = __ldg(reinterpret_cast<const float4 *>(p.A + static_cast<long long>(ga_row) * p.lda + ka));
      }
      if (OPB) {
        if (gb_col < p.N && kb < p.K)
          vb = __ldg(reinterpret_cast<const float4 *>(p.B + static_cast<long long>(gb_col) * p.ldb + kb));
      } else if (kb < p.K && gb_col < p.N) {
        vb = __ldg(reinterpret_cast<const float4 *>(p.B + static_cast<long long>(kb) * p.ldb + gb_col));
      }
      a_reg[0] = va.x; a_reg[1] = va.y; a_reg[2] = va.z; a_reg[3] = va.w;
      b_reg[0] = vb.x; b_reg[1] = vb.y; b_reg[2] = vb.z; b_reg[3] = vb.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (OPA)
          a_reg[j] = (ka < p.K && ga_row + j < p.M)
                         ? __ldg(p.A + static_cast<long long>(ka) * p.lda + ga_row + j)
                         : 0.0f;
        else
          a_reg[j] = (ga_row < p.M && ka + j < p.K)
                         ? __ldg(p.A + static_cast<long long>(ga_row) * p.lda + ka + j)
                         : 0.0f;
        if (OPB)
          b_reg[j] = (gb_col < p.N && kb + j < p.K)
                         ? __ldg(p.B + static_cast<long long>(gb_col) * p.ldb + kb + j)
                         : 0.0f;
        else
          b_reg[j] = (kb < p.K && gb_col + j < p.N)
                         ? __ldg(p.B + static_cast<long long>(kb) * p.ldb + gb_col + j)
                         : 0.0f;
      }
    }
  };
  auto store_slice = [&](int buf) {
    if (OPA) {
      *reinterpret_cast<float4 *>(&As[buf][a_k][a_row]) =
          make_float4(a_reg[0], a_reg[1], a_reg[2], a_reg[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) As[buf][a_k + j][a_row] = a_reg[j];
    }
    if (OPB) {
#pragma unroll
      for (int j = 0; j < 4; ++j) Bs[buf][b_k + j][b_col] = b_reg[j];
    } else {
      *reinterpret_cast<float4 *>(&Bs[buf][b_k][b_col]) =
          make_float4(b_reg[0], b_reg[1], b_reg[2], b_reg[3]);
    }
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
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = p.alpha * acc[i][h * 4 + j];
      if (VEC) {
        if (col < p.N) {
          float4 *dst = reinterpret_cast<float4 *>(crow + col);
          if (p.beta != 0.0f) {
            const float4 c = *dst;
            v[0] += p.beta * c.x;
            v[1] += p.beta * c.y;
            v[2] += p.beta * c.z;
            v[3] += p.beta * c.w;
          }
          *dst = make_float4(v[0], v[1], v[2], v[3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (col + j < p.N) {
            if (p.beta != 0.0f) v[j] += p.beta * crow[col + j];
            crow[col + j] = v[j];
          }
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
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.tiles_m = static_cast<int>((a.M + kTile - 1) / kTile);
  p.tiles_n = static_cast<int>((a.N + kTile - 1) / kTile);
  const long long blocks = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (blocks > 0x7fffffffLL) return kErrInvalidArg;
  // 128-bit accesses: every pointer 16-byte aligned, every pitch and every
  // contiguous extent (A: K, or M when stored transposed; B: N, or K; C: N) a
  // multiple of 4, so a 4-wide group is wholly inside or outside.
  const int64_t a_inner = a.opa ? a.M : a.K, b_inner = a.opb ? a.K : a.N;
  const bool vec = reinterpret_cast<uintptr_t>(a.A) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.B) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.lda % 4 == 0 &&
                   a.ldb % 4 == 0 && a.ldc % 4 == 0 && a_inner % 4 == 0 && b_inner % 4 == 0 &&
                   a.N % 4 == 0;
  const dim3 grid(static_cast<unsigned>(blocks));
  const int variant = (vec ? 4 : 0) | (a.opb ? 2 : 0) | (a.opa ? 1 : 0);
  switch (variant) {
    case 0: simt_gemm_kernel<false, false, false><<<grid, kThreads, 0, stream>>>(p); break;
    case 1: simt_gemm_kernel<false, false, true><<<grid, kThreads, 0, stream>>>(p); break;
    case 2: simt_gemm_kernel<false, true, false><<<grid, kThreads, 0, stream>>>(p); break;
    case 3: simt_gemm_kernel<false, true, true><<<grid, kThreads, 0, stream>>>(p); break;
    case 4: simt_gemm_kernel<true, false, false><<<grid, kThreads, 0, stream>>>(p); break;
    case 5: simt_gemm_kernel<true, false, true><<<grid, kThreads, 0, stream>>>(p); break;
    case 6: simt_gemm_kernel<true, true, false><<<grid, kThreads, 0, stream>>>(p); break;
    default: simt_gemm_kernel<true, true, true><<<grid, kThreads, 0, stream>>>(p); break;
  }
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace gemm
