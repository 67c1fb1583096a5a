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
//   * K advances in slices of 32 through two shared-memory stages filled by
//     asynchronous copies (cp.async), so the copies of slice s + 1 run while
//     slice s is multiplied and no register holds operand data in flight. A
//     is staged transposed (k-major, rows padded to 132 floats): each lane
//     copies one 4-byte element into its transposed place, eight lanes per
//     row so that a warp reads 32-byte row segments and writes 32 distinct
//     banks. B, and A when it is stored K x M, are copied as they are, 16
//     bytes per copy when the operands allow (VEC), else 4;
//   * elements outside the matrices are zero-filled by the copies (source
//     size 0) and every store is guarded, the boundary rule of section 4 of
//     "WebGPU WGSL Compute Shaders: Custom Matrix Multiplication (GEMM)
//     Optimization Guide".
//
// Each output is accumulated by fused multiply-adds over k in increasing
// order in fp32, so |C - AB| <= K 2^-24 |A||B| element-wise. The general form
// C = alpha * A op(B) + beta * C scales the sum once at the store (C is read
// only when beta != 0). op(B) = B, or B stored transposed (N x K, the vec4
// transposed-B storage of the subgroups page, section 7), which is staged
// through the same transposing copies as A; op(A) = A, or A stored
// transposed (K x M), whose rows of m are copied into the k-major tile as is.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace gemm {
namespace {

constexpr int kTile = 128;
constexpr int kSliceK = 32;                  // k per stage
constexpr int kThreads = 256;
constexpr int kPitch = kTile + 4;            // floats per k-row of a stage tile
constexpr int kStageFloats = 2 * kSliceK * kPitch;  // A tile + B tile
constexpr int kSmemBytes = 2 * kStageFloats * 4;    // two stages: 67,584 bytes
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
  // Extents in elements of A, B and C for the checked build's index checks.
  long long a_extent, b_extent, c_extent;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Asynchronous copy of 4 (or 16) bytes into shared memory; when `in` is
// false nothing is read and the destination is zero-filled.
__device__ __forceinline__ void copy4(uint32_t dst, const float *src, bool in) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
               "r"(in ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void copy16(uint32_t dst, const float *src, bool in) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(in ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void copy_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void copy_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

template <bool VEC, bool OPB, bool OPA>
__global__ void __launch_bounds__(kThreads, 2) simt_gemm_kernel(const SimtParams p) {
  extern __shared__ __align__(16) float smem[];

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
  const int lane = tid & 31, warp = tid >> 5;
  const int tx = tid & 15, ty = tid >> 4;
  const uint32_t sbase = smem_addr(smem);

  // Copies of slice s (k0 = s * kSliceK) into stage s & 1, in groups of 8 k.
  // Transposing copies (A stored M x K, B stored N x K): lane -> row
  // warp * 16 + j * 4 + lane / 8, k lane % 8. Direct copies (A stored K x M,
  // B stored K x N): k-row tid / 32, columns (tid % 32) * 4 ... + 3 (VEC) or
  // tid % 32 + 32 j.
  auto issue = [&](int s) {
    const uint32_t as = sbase + (s & 1) * kStageFloats * 4;
    const uint32_t bs = as + kSliceK * kPitch * 4;
#pragma unroll
    for (int h = 0; h < kSliceK / 8; ++h) {
      const int k0 = s * kSliceK + h * 8;
      if constexpr (!OPA) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = warp * 16 + j * 4 + (lane >> 3), kk = lane & 7;
          const long long off = static_cast<long long>(m0 + row) * p.lda + k0 + kk;
          const bool in = m0 + row < p.M && k0 + kk < p.K &&
                          index_ok(kSiteLoadA, off, 1, p.a_extent);
          const float *src = in ? p.A + off : p.A;
          copy4(as + ((h * 8 + kk) * kPitch + row) * 4, src, in);
        }
      } else if constexpr (VEC) {
        const int kk = tid >> 5, col = lane * 4;
        const long long off = static_cast<long long>(k0 + kk) * p.lda + m0 + col;
        const bool in = k0 + kk < p.K && m0 + col < p.M &&
                        index_ok(kSiteLoadA, off, 4, p.a_extent);
        const float *src = in ? p.A + off : p.A;
        copy16(as + ((h * 8 + kk) * kPitch + col) * 4, src, in);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kk = tid >> 5, col = lane + 32 * j;
          const long long off = static_cast<long long>(k0 + kk) * p.lda + m0 + col;
          const bool in = k0 + kk < p.K && m0 + col < p.M &&
                          index_ok(kSiteLoadA, off, 1, p.a_extent);
          const float *src = in ? p.A + off : p.A;
          copy4(as + ((h * 8 + kk) * kPitch + col) * 4, src, in);
        }
      }
      if constexpr (OPB) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = warp * 16 + j * 4 + (lane >> 3), kk = lane & 7;
          const long long off = static_cast<long long>(n0 + col) * p.ldb + k0 + kk;
          const bool in = n0 + col < p.N && k0 + kk < p.K &&
                          index_ok(kSiteLoadB, off, 1, p.b_extent);
          const float *src = in ? p.B + off : p.B;
          copy4(bs + ((h * 8 + kk) * kPitch + col) * 4, src, in);
        }
      } else if constexpr (VEC) {
        const int kk = tid >> 5, col = lane * 4;
        const long long off = static_cast<long long>(k0 + kk) * p.ldb + n0 + col;
        const bool in = k0 + kk < p.K && n0 + col < p.N &&
                        index_ok(kSiteLoadB, off, 4, p.b_extent);
        const float *src = in ? p.B + off : p.B;
        copy16(bs + ((h * 8 + kk) * kPitch + col) * 4, src, in);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kk = tid >> 5, col = lane + 32 * j;
          const long long off = static_cast<long long>(k0 + kk) * p.ldb + n0 + col;
          const bool in = k0 + kk < p.K && n0 + col < p.N &&
                          index_ok(kSiteLoadB, off, 1, p.b_extent);
          const float *src = in ? p.B + off : p.B;
          copy4(bs + ((h * 8 + kk) * kPitch + col) * 4, src, in);
        }
      }
    }
    copy_commit();
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  const int num_slices = (p.K + kSliceK - 1) / kSliceK;
  issue(0);
  for (int s = 0; s < num_slices; ++s) {
    // Slice s has landed (this thread's copies, then everyone's), and every
    // thread is done with slice s - 1, whose stage the next copies refill.
    copy_wait_all();
    __syncthreads();
    if (s + 1 < num_slices) issue(s + 1);
    const float *As = smem + (s & 1) * kStageFloats;
    const float *Bs = As + kSliceK * kPitch;
    // Unrolled by 4 only: the whole 32-k slice unrolled (2,000+ instructions)
    // no longer fits the instruction cache and runs 2-3 % slower.
#pragma unroll 4
    for (int k = 0; k < kSliceK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&As[k * kPitch + ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&As[k * kPitch + 64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[k * kPitch + tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[k * kPitch + 64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
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
        if (col < p.N && ptr_ok(kSiteCStore, crow + col, 4, p.C, p.c_extent)) {
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
          if (col + j < p.N && ptr_ok(kSiteCStore, crow + col + j, 1, p.C, p.c_extent)) {
            if (p.beta != 0.0f) v[j] += p.beta * crow[col + j];
            crow[col + j] = v[j];
          }
      }
    }
  }
}

// Launch one variant; its shared memory (above the 48 KiB default) is
// enabled once per device.
template <bool VEC, bool OPB, bool OPA>
int launch_variant(const SimtParams &p, dim3 grid, cudaStream_t stream) {
  auto kernel = simt_gemm_kernel<VEC, OPB, OPA>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kErrLaunch;
  static bool attr_set[64] = {};
  static std::mutex attr_mu;
  {
    std::lock_guard<std::mutex> g(attr_mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
          cudaSuccess)
        return kErrLaunch;
      attr_set[dev] = true;
    }
  }
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrLaunch;
}

}  // namespace

GEMM_INDEX_FAULT_TAKE(simt_index_fault_take)

// 128-bit accesses: every pointer 16-byte aligned, every pitch and every
// contiguous extent (A: K, or M when stored transposed; B: N, or K; C: N) a
// multiple of 4, so a 4-wide group is wholly inside or outside.
bool simt_vec_ok(const GemmArgs &a) {
  const int64_t a_inner = a.opa ? a.M : a.K, b_inner = a.opb ? a.K : a.N;
  return reinterpret_cast<uintptr_t>(a.A) % 16 == 0 && reinterpret_cast<uintptr_t>(a.B) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.lda % 4 == 0 && a.ldb % 4 == 0 &&
         a.ldc % 4 == 0 && a_inner % 4 == 0 && b_inner % 4 == 0 && a.N % 4 == 0;
}

int simt_launch_direct(const GemmArgs &a, cudaStream_t stream) {
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
  p.a_extent = a.opa ? matrix_extent(a.K, a.M, a.lda) : matrix_extent(a.M, a.K, a.lda);
  p.b_extent = a.opb ? matrix_extent(a.N, a.K, a.ldb) : matrix_extent(a.K, a.N, a.ldb);
  p.c_extent = c_extent_of(a);
  p.tiles_m = static_cast<int>((a.M + kTile - 1) / kTile);
  p.tiles_n = static_cast<int>((a.N + kTile - 1) / kTile);
  const long long blocks = static_cast<long long>(p.tiles_m) * p.tiles_n;
  if (blocks > 0x7fffffffLL) return kErrInvalidArg;
  const bool vec = simt_vec_ok(a);
  const dim3 grid(static_cast<unsigned>(blocks));
  const int variant = (vec ? 4 : 0) | (a.opb ? 2 : 0) | (a.opa ? 1 : 0);
  switch (variant) {
    case 0: return launch_variant<false, false, false>(p, grid, stream);
    case 1: return launch_variant<false, false, true>(p, grid, stream);
    case 2: return launch_variant<false, true, false>(p, grid, stream);
    case 3: return launch_variant<false, true, true>(p, grid, stream);
    case 4: return launch_variant<true, false, false>(p, grid, stream);
    case 5: return launch_variant<true, false, true>(p, grid, stream);
    case 6: return launch_variant<true, true, false>(p, grid, stream);
    default: return launch_variant<true, true, true>(p, grid, stream);
  }
}

int simt_launch(const GemmArgs &a, int sm_count, bool may_alloc, cudaStream_t stream) {
  // A stored M x K is staged by sixteen transposing 4-byte copies per thread
  // and 32-k slice; stored K x M, by four 16-byte copies with no bank
  // conflicts: 2364 against 2522 us at 4096^3. Transposing A first (into a
  // workspace from the library's pool; about 20 us at 4096^3) pays once N is
  // large, the transpose's share falling as 1 / N: from N = 1024, when the
  // transposed call keeps the 16-byte path. Results are the same: each
  // output is accumulated over k in the same order either way.
  if (may_alloc && !a.opa && a.N >= 1024 && a.K >= 64 && a.M % 4 == 0) {
    GemmArgs t = a;
    t.opa = 1;
    t.lda = a.M;
    t.A = reinterpret_cast<const float *>(uintptr_t{256});  // a pool block's alignment
    if (simt_vec_ok(t)) {
      void *ws = nullptr;
      int st = pool_alloc(&ws, static_cast<size_t>(a.K) * a.M * 4, stream);
      if (st != kOk) return st;
      float *at = static_cast<float *>(ws);
      t.A = at;
      st = transpose_launch(a.A, a.lda, a.M, a.K, at, a.M, sm_count, stream);
      if (st == kOk) st = simt_launch_direct(t, stream);
      const int fst = pool_free(ws, stream);
      return st != kOk ? st : fst;
    }
  }
  return simt_launch_direct(a, stream);
}

}  // namespace gemm
