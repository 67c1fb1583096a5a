// tc_gemm.cu -- tensor-core fp32 GEMM for sm_103a (tcgen05 + TMEM).
//
// C[M x N] = A[M x K] * B[K x N], all row-major fp32.
//
// Formulation. kind::tf32 MMAs need both operands K-major (k contiguous). A
// (row-major M x K) already is; B (row-major K x N) is N-contiguous. Each
// output tile is therefore computed transposed,
//
//     D = C_tile^T  (128 n x 256 m)  =  B_tile^T (128 n x K)  *  A_tile^T (K x 256 m),
//
// with B_tile^T as the MMA's A operand held in TMEM (lane = n, one 32-bit
// column per k: the transpose happens on the way from shared memory through
// registers into TMEM) and the A tile, staged K-major by TMA, as the MMA's B
// operand in shared memory. The accumulator D lives in TMEM with lane = n and
// column = m, so each epilogue store writes 32 consecutive columns of one row
// of C (a coalesced 128-byte segment).
//
// Roles (warp-specialised, persistent, one CTA per SM, grouped raster):
//   producer   TMA: one thread loads the 256 x 32 A tile (128-byte swizzle)
//              and the 32 x 128 B tile per stage into a ring of stages.
//              LSU (operands TMA cannot describe): four warps load both with
//              plain loads and place the A tile in shared memory and B^T in
//              TMEM themselves.
//   transform  (TMA variant) four warps move B^T into TMEM and, in 3xTF32
//              mode, split the A tile into hi (in place) and lo (sibling tile).
//   MMA        one thread issues tcgen05.mma kind::tf32, M = 128, N = 256,
//              K = 8. 3xTF32 issues B_lo*A_hi, B_hi*A_lo, B_hi*A_hi per k-step
//              (small terms first), hi = tf32(x), lo = tf32(x - hi).
//   epilogue   four warps read D from TMEM and store C with row/column
//              guards.
//
// This is the tiled product of "Optimizing a WebGPU Matmul Kernel using
// Subgroups" (sections 4-8: shared-memory tiles, register tiles, vector
// loads, matrix-unit multiply-accumulate over staged tiles, output staged
// before the store) mapped onto Blackwell's tensor memory and copy engine;
// out-of-range elements load as zero and stores are guarded, as in section 4
// of "WebGPU WGSL Compute Shaders: Custom Matrix Multiplication (GEMM)
// Optimization Guide". Section 6 of that guide transposes a shared-memory
// tile to avoid bank conflicts; here the transpose of B is what makes the
// operand K-major for the tensor core.
//
// Every barrier wait is bounded (mbar_wait_bounded). On a timeout the CTA
// lets its in-flight copies and MMAs finish (bounded), frees TMEM and exits;
// the host reads kErrTimeout from the status word.

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"

namespace gemm {

__device__ int g_tc_status;  // first error recorded by any kernel of this unit

namespace {

constexpr int kTM = 256;        // rows of C per tile   (MMA N)
constexpr int kTN = 128;        // columns of C per tile (MMA M = TMEM lanes)
constexpr int kBK = 32;         // K per stage: 32 fp32 = one 128-byte swizzle row of A
constexpr int kUmmaK = 8;       // K per tcgen05.mma of kind::tf32
constexpr int kGroupM = 8;      // m-blocks per raster group
constexpr uint32_t kSw128 = 2;  // descriptor layout type: 128-byte swizzle
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;    // D: columns [0, 256)
constexpr uint32_t kBtCol = 256;   // B^T stage buffers from column 256

struct TcParams {
  int M, N, K;
  const float *A;
  long long lda;
  const float *B;
  long long ldb;
  float *C;
  long long ldc;
  int num_m_blocks, num_n_blocks, num_tiles, num_k_blocks;
  unsigned long long timeout_ns;
};

template <int STAGES, bool EXACT, bool LSU>
struct TcConfig {
  static constexpr int kABytes = kTM * kBK * 4;                  // 32 KiB, K-major, swizzled
  static constexpr int kBBytes = LSU ? 0 : kBK * kTN * 4;        // 16 KiB, row-major (TMA)
  static constexpr int kALoBytes = EXACT ? kABytes : 0;          // 3xTF32 lo tile of A
  static constexpr int kStageBytes = kABytes + kBBytes + kALoBytes;
  static constexpr int kBOffset = kABytes;
  static constexpr int kALoOffset = kABytes + kBBytes;
  static constexpr int kTileBytes = STAGES * kStageBytes;
  static constexpr uint32_t kBtColsPerStage = EXACT ? 2 * kBK : kBK;  // hi (+ lo)
  static constexpr int kProdWarps = LSU ? 4 : 1;
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kEpiWarp0 = kMmaWarp + 1;
  static constexpr int kXformWarps = LSU ? 0 : 4;
  static constexpr int kXformWarp0 = kEpiWarp0 + 4;
  static constexpr int kThreads = 32 * (kXformWarp0 + kXformWarps);
  static constexpr uint32_t kIdesc = idesc_tf32(kTN, kTM);
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kBtCol + STAGES * kBtColsPerStage <= kTmemCols, "TMEM budget");
};

template <int STAGES>
struct alignas(8) TcShared {
  uint64_t full[STAGES];   // stage loaded (TMA bytes, or the LSU producer warps)
  uint64_t ready[STAGES];  // B^T in TMEM (and A split) by the transform warps
  uint64_t empty[STAGES];  // stage consumed by the MMAs (tcgen05.commit)
  uint64_t acc_full;       // accumulator complete (tcgen05.commit)
  uint64_t acc_empty;      // accumulator drained by the epilogue warps
  uint64_t drain;          // every MMA of this CTA has completed
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void tile_coords(const TcParams &p, int t, int &mb, int &nb) {
  const int group_tiles = kGroupM * p.num_n_blocks;
  const int g = t / group_tiles;
  const int first_m = g * kGroupM;
  const int gm = min(p.num_m_blocks - first_m, kGroupM);
  const int r = t - g * group_tiles;
  mb = first_m + r % gm;
  nb = r / gm;
}

// 128-byte swizzle inside 1024-byte groups of eight 128-byte rows: the
// 16-byte chunk index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t sw128(uint32_t linear) {
  return linear ^ (((linear >> 7) & 7u) << 4);
}

// Wait with a warp-uniform outcome (every lane of the warp waits).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const TcParams &p,
                                          volatile int *abort) {
  const bool ok = mbar_wait_bounded(bar, parity, p.timeout_ns, abort, &g_tc_status);
  return __all_sync(0xffffffffu, ok);
}

// Spin (bounded, ignoring the abort flag) until the phase completes.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) break;
  }
}

// 32 values of B^T row n (k = 0..31 of the stage) into TMEM, raw or as the
// 3xTF32 pair hi = tf32(x), lo = tf32(x - hi).
template <bool EXACT>
__device__ __forceinline__ void bt_to_tmem(uint32_t t_hi, uint32_t t_lo, const float (&v)[32]) {
  uint32_t hi[32];
  if (EXACT) {
    uint32_t lo[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float h = round_tf32(v[k]);
      hi[k] = __float_as_uint(h);
      lo[k] = __float_as_uint(round_tf32(v[k] - h));
    }
    tmem_store_32cols(t_hi, hi);
    tmem_store_32cols(t_lo, lo);
  } else {
#pragma unroll
    for (int k = 0; k < 32; ++k) hi[k] = __float_as_uint(v[k]);
    tmem_store_32cols(t_hi, hi);
  }
}

template <bool EXACT>
__device__ __forceinline__ void stage_a_value(uint8_t *stage, int lo_offset, uint32_t off,
                                              float v) {
  if (EXACT) {
    const float hi = round_tf32(v);
    *reinterpret_cast<float *>(stage + off) = hi;
    *reinterpret_cast<float *>(stage + lo_offset + off) = round_tf32(v - hi);
  } else {
    *reinterpret_cast<float *>(stage + off) = v;
  }
}

template <int STAGES, bool EXACT, bool LSU>
__global__ void __launch_bounds__(TcConfig<STAGES, EXACT, LSU>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const TcParams p) {
  using Cfg = TcConfig<STAGES, EXACT, LSU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcShared<STAGES> *sh = reinterpret_cast<TcShared<STAGES> *>(tiles + Cfg::kTileBytes);
  volatile int *abort = &sh->abort;

  const uint32_t warp = warp_index();
  const uint32_t lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full[s], LSU ? Cfg::kProdWarps : 1);
      mbar_init(&sh->ready[s], Cfg::kXformWarps > 0 ? Cfg::kXformWarps : 1);
      mbar_init(&sh->empty[s], 1);
    }
    mbar_init(&sh->acc_full, 1);
    mbar_init(&sh->acc_empty, 4);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
  }
  if (!LSU && warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem_base;

  if (!LSU && warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_parity = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          if (!mbar_wait_bounded(&sh->empty[stage], phase ^ 1, p.timeout_ns, abort,
                                 &g_tc_status)) {
            ok = false;
            break;
          }
          uint8_t *st = tiles + stage * Cfg::kStageBytes;
          mbar_arrive_expect_tx(&sh->full[stage], Cfg::kABytes + kBK * kTN * 4);
          tma_load_2d(st, &tmap_a, &sh->full[stage], kb * kBK, mb * kTM);
          tma_load_2d(st + Cfg::kBOffset, &tmap_b, &sh->full[stage], nb * kTN, kb * kBK);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // Let every TMA copy this thread issued land before the CTA exits.
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) drain_wait(&sh->full[s], (armed_parity >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (LSU && warp < Cfg::kProdWarps) {
    // ------------------------------------------------------ LSU producer --
    // Warp w stages A rows w, w + 4, ... (lane = k) and B^T rows
    // n = 32 w + lane (TMEM lanes of this warp's quadrant).
    uint32_t stage = 0, phase = 0;
    const uint32_t quad = warp & 3;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m0 = mb * kTM, n0 = nb * kTN;
      bool ok = true;
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        if (!warp_wait(&sh->empty[stage], phase ^ 1, p, abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint8_t *st = tiles + stage * Cfg::kStageBytes;
        const int k0 = kb * kBK;
        const int gk = k0 + lane;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int gm = m0 + warp + 4 * (half * 32 + i);
            v[i] = (gm < p.M && gk < p.K) ? __ldg(p.A + static_cast<long long>(gm) * p.lda + gk)
                                          : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            stage_a_value<EXACT>(st, Cfg::kALoOffset,
                                 sw128((warp + 4 * (half * 32 + i)) * 128 + lane * 4), v[i]);
        }
        {
          const int gn = n0 + quad * 32 + lane;
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k)
            v[k] = (gn < p.N && k0 + k < p.K)
                       ? __ldg(p.B + static_cast<long long>(k0 + k) * p.ldb + gn)
                       : 0.0f;
          const uint32_t col = tmem + ((quad * 32) << 16) + kBtCol + stage * Cfg::kBtColsPerStage;
          bt_to_tmem<EXACT>(col, col + kBK, v);
        }
        fence_proxy_async_smem();
        tmem_store_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->full[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
    }
  } else if (warp == Cfg::kMmaWarp) {
    // -------------------------------------------------------------- MMA --
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t d_tmem = tmem + kAccCol;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!mbar_wait_bounded(&sh->acc_empty, acc_phase ^ 1, p.timeout_ns, abort,
                               &g_tc_status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          uint64_t *in_bar = LSU ? &sh->full[stage] : &sh->ready[stage];
          if (!mbar_wait_bounded(in_bar, phase, p.timeout_ns, abort, &g_tc_status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_hi = smem_addr(tiles + stage * Cfg::kStageBytes);
          const uint32_t bt_hi = tmem + kBtCol + stage * Cfg::kBtColsPerStage;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            // A tile, K-major: a k-step of 8 fp32 is 32 bytes along the swizzled row;
            // 8-row groups are 1024 bytes apart.
            const uint64_t da = smem_desc(a_hi + kk * 32, 16, 1024, kSw128);
            const uint32_t accumulate = (kb | kk) != 0;
            if (EXACT) {
              const uint64_t da_lo = smem_desc(a_hi + Cfg::kALoOffset + kk * 32, 16, 1024, kSw128);
              mma_tf32_ts(d_tmem, bt_hi + kBK + kk * kUmmaK, da, Cfg::kIdesc, accumulate);
              mma_tf32_ts(d_tmem, bt_hi + kk * kUmmaK, da_lo, Cfg::kIdesc, 1);
              mma_tf32_ts(d_tmem, bt_hi + kk * kUmmaK, da, Cfg::kIdesc, 1);
            } else {
              mma_tf32_ts(d_tmem, bt_hi + kk * kUmmaK, da, Cfg::kIdesc, accumulate);
            }
          }
          mma_commit(&sh->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&sh->acc_full);
        acc_phase ^= 1;
      }
      // Every MMA this thread issued completes before TMEM is released.
      mma_commit(&sh->drain);
      drain_wait(&sh->drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= Cfg::kEpiWarp0 && warp < Cfg::kEpiWarp0 + 4) {
    // --------------------------------------------------------- epilogue --
    const uint32_t quad = warp & 3;  // TMEM lanes (columns of C) this warp may read
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      if (!warp_wait(&sh->acc_full, acc_phase, p, abort)) break;
      tc_fence_after_sync();
      const int gn = nb * kTN + quad * 32 + lane;
      const bool n_ok = gn < p.N;
      const uint32_t t_lane = tmem + ((quad * 32) << 16) + kAccCol;
#pragma unroll 1
      for (int c = 0; c < kTM / 32; ++c) {
        const int gm0 = mb * kTM + c * 32;
        if (gm0 >= p.M) break;
        uint32_t r[32];
        tmem_load_32cols(t_lane + c * 32, r);
        tmem_load_wait();
        float *dst = p.C + static_cast<long long>(gm0) * p.ldc + gn;
        const int rows = min(32, p.M - gm0);
        if (n_ok) {
          if (rows == 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[static_cast<long long>(j) * p.ldc] = __uint_as_float(r[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < rows) dst[static_cast<long long>(j) * p.ldc] = __uint_as_float(r[j]);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty);
      acc_phase ^= 1;
    }
  } else if (Cfg::kXformWarps > 0 && warp >= Cfg::kXformWarp0) {
    // -------------------------------------------- transform (TMA variant) --
    const uint32_t quad = warp & 3;
    const int xt = threadIdx.x - Cfg::kXformWarp0 * 32;  // 0..127
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        if (!warp_wait(&sh->full[stage], phase, p, abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint8_t *st = tiles + stage * Cfg::kStageBytes;
        {
          // B tile is row-major 32 k x 128 n (512-byte rows); this thread's
          // column n = 32 quad + lane becomes TMEM lane n.
          const float *bs = reinterpret_cast<const float *>(st + Cfg::kBOffset) + quad * 32 + lane;
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = bs[k * kTN];
          const uint32_t col = tmem + ((quad * 32) << 16) + kBtCol + stage * Cfg::kBtColsPerStage;
          bt_to_tmem<EXACT>(col, col + kBK, v);
        }
        if (EXACT) {
          float4 *raw = reinterpret_cast<float4 *>(st);
          float4 *lo = reinterpret_cast<float4 *>(st + Cfg::kALoOffset);
#pragma unroll 4
          for (int i = xt; i < Cfg::kABytes / 16; i += 32 * Cfg::kXformWarps) {
            const float4 x = raw[i];
            float4 h, l;
            h.x = round_tf32(x.x);
            h.y = round_tf32(x.y);
            h.z = round_tf32(x.z);
            h.w = round_tf32(x.w);
            l.x = round_tf32(x.x - h.x);
            l.y = round_tf32(x.y - h.y);
            l.z = round_tf32(x.z - h.z);
            l.w = round_tf32(x.w - h.w);
            raw[i] = h;
            lo[i] = l;
          }
          fence_proxy_async_smem();
        }
        tmem_store_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->ready[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One warp waits, bounded, on a barrier that is never signalled.
__global__ void selftest_wait_kernel(unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait_bounded(&bar, 0, timeout_ns, &abort_flag, &g_tc_status);
}

// ------------------------------------------------------------------ host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Small cache of encoded tensor maps keyed by (address, extents, pitch, box, swizzle).
struct MapKey {
  const void *ptr;
  uint64_t d0, d1, pitch;
  uint32_t b0, b1, swizzle;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && pitch == o.pitch && b0 == o.b0 &&
           b1 == o.b1 && swizzle == o.swizzle;
  }
};

struct MapCache {
  static constexpr int kSlots = 32;
  MapKey keys[kSlots];
  CUtensorMap maps[kSlots];
  bool used[kSlots] = {};
  int next = 0;
  std::mutex mu;
};

// 2-D fp32 tensor map over a row-major matrix (d0 = columns, d1 = rows) with a
// b0 x b1 box, the given swizzle, and zero fill outside the matrix.
bool get_map(const void *ptr, uint64_t d0, uint64_t d1, uint64_t pitch_bytes, uint32_t b0,
             uint32_t b1, CUtensorMapSwizzle swizzle, CUtensorMap *out) {
  static MapCache cache;
  const MapKey key{ptr, d0, d1, pitch_bytes, b0, b1, static_cast<uint32_t>(swizzle)};
  {
    std::lock_guard<std::mutex> g(cache.mu);
    for (int i = 0; i < MapCache::kSlots; ++i)
      if (cache.used[i] && cache.keys[i] == key) {
        *out = cache.maps[i];
        return true;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {b0, b1};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> g(cache.mu);
  const int slot = cache.next;
  cache.next = (cache.next + 1) % MapCache::kSlots;
  cache.keys[slot] = key;
  cache.maps[slot] = m;
  cache.used[slot] = true;
  *out = m;
  return true;
}

template <int STAGES, bool EXACT, bool LSU>
int launch_variant(const GemmArgs &a, int sm_count, cudaStream_t stream) {
  using Cfg = TcConfig<STAGES, EXACT, LSU>;
  auto kernel = tc_gemm_kernel<STAGES, EXACT, LSU>;
  const int smem_bytes = Cfg::kTileBytes + static_cast<int>(sizeof(TcShared<STAGES>)) + 1024;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kErrLaunch;
  static bool attr_set[64] = {};
  static std::mutex attr_mu;
  {
    std::lock_guard<std::mutex> g(attr_mu);
    if (dev < 64 && !attr_set[dev]) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
          cudaSuccess)
        return kErrLaunch;
      attr_set[dev] = true;
    }
  }

  CUtensorMap map_a, map_b;
  std::memset(&map_a, 0, sizeof(map_a));
  std::memset(&map_b, 0, sizeof(map_b));
  if (!LSU) {
    if (!get_map(a.A, a.K, a.M, a.lda * 4, kBK, kTM, CU_TENSOR_MAP_SWIZZLE_128B, &map_a))
      return kErrLaunch;
    if (!get_map(a.B, a.N, a.K, a.ldb * 4, kTN, kBK, CU_TENSOR_MAP_SWIZZLE_NONE, &map_b))
      return kErrLaunch;
  }

  TcParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.A = a.A;
  p.lda = a.lda;
  p.B = a.B;
  p.ldb = a.ldb;
  p.C = a.C;
  p.ldc = a.ldc;
  p.num_m_blocks = static_cast<int>((a.M + kTM - 1) / kTM);
  p.num_n_blocks = static_cast<int>((a.N + kTN - 1) / kTN);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  p.num_k_blocks = static_cast<int>((a.K + kBK - 1) / kBK);
  // Generous: a stage takes microseconds; one tile's mainloop about K * 25 ns.
  p.timeout_ns = 2000000000ull + static_cast<unsigned long long>(a.K) * 2000ull;

  const int grid = p.num_tiles < sm_count ? p.num_tiles : sm_count;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  if (cudaLaunchKernelEx(&cfg, kernel, map_a, map_b, p) != cudaSuccess) return kErrLaunch;
  return kOk;
}

}  // namespace

bool tc_tma_legal(const GemmArgs &a) {
  return reinterpret_cast<uintptr_t>(a.A) % 16 == 0 && reinterpret_cast<uintptr_t>(a.B) % 16 == 0 &&
         a.lda % 4 == 0 && a.ldb % 4 == 0;
}

int tc_launch(const GemmArgs &a, bool exact, bool lsu, int sm_count, cudaStream_t stream) {
  if (exact) {
    if (lsu) return launch_variant<2, true, true>(a, sm_count, stream);
    return launch_variant<2, true, false>(a, sm_count, stream);
  }
  if (lsu) return launch_variant<4, false, true>(a, sm_count, stream);
  return launch_variant<4, false, false>(a, sm_count, stream);
}

int tc_poll_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return kErrLaunch;
  int h = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&h, g_tc_status, sizeof(int)) != cudaSuccess) return kErrLaunch;
  if (h != 0 && cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess)
    return kErrLaunch;
  return h;
}

int tc_selftest_wait_timeout(int64_t timeout_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(timeout_ns));
  if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
  return tc_poll_status(stream);
}

}  // namespace gemm
