// tc_gemm.cu -- tensor-core fp32 GEMM for sm_103a (tcgen05 + TMEM).
//
// C[M x N] = A[M x K] * B[K x N], all row-major fp32. One persistent CTA per
// SM walks a grouped (L2-friendly) sequence of 128 x BN output tiles. Roles
// are warp-specialised and talk through mbarriers:
//
//   producer  stages 128 x 32 tiles of A and 32 x BN tiles of B into a ring of
//             shared-memory stages in the 128-byte swizzled layouts tcgen05
//             reads: either one thread issuing TMA tile loads (TMA-legal
//             operands) or four warps issuing plain loads (any strides).
//   transform (3xTF32 with TMA only) splits every staged value x into
//             hi = tf32(x) and lo = tf32(x - hi), hi in place, lo in a
//             sibling tile at the same offset.
//   MMA       one thread issues tcgen05.mma kind::tf32 (M = 128, N = BN,
//             K = 8) into a TMEM accumulator; 3xTF32 issues A_lo*B_hi,
//             A_hi*B_lo, A_hi*B_hi per k-step (small terms first). Two TMEM
//             accumulators let the epilogue of one tile overlap the mainloop
//             of the next.
//   epilogue  four warps move the accumulator TMEM -> registers -> global
//             memory with row/column predication.
//
// This is the tiled product of "Optimizing a WebGPU Matmul Kernel using
// Subgroups" (sections 4-8: shared-memory tiles, per-thread register tiles,
// vector loads, matrix-unit multiply-accumulate over staged tiles, output
// staged before the store) mapped onto Blackwell's tensor memory and async
// copy engine; the zero-filled out-of-range loads and guarded stores are
// those of section 4 of "WebGPU WGSL Compute Shaders: Custom Matrix
// Multiplication (GEMM) Optimization Guide".
//
// Every barrier wait is bounded (see mbar_wait_bounded); on a timeout the CTA
// drains its in-flight copies and MMAs, frees TMEM and exits, and the host
// reads kErrTimeout from the status word.

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

constexpr int kBM = 128;       // rows of A / C per tile (= TMEM lanes)
constexpr int kBK = 32;        // K per stage: 32 fp32 = one 128-byte swizzle row
constexpr int kUmmaK = 8;      // K per tcgen05.mma of kind::tf32
constexpr int kGroupM = 8;     // m-blocks per raster group
constexpr uint32_t kSw128 = 2; // descriptor layout type: 128-byte swizzle

struct TcParams {
  int M, N, K;
  const float *A;
  long long lda;
  const float *B;
  long long ldb;
  float *C;
  long long ldc;
  int num_m_blocks, num_n_blocks, num_tiles, num_k_blocks;
  int vec_store;  // C 16-byte aligned and ldc % 4 == 0
  unsigned long long timeout_ns;
};

template <int BN, int STAGES, bool EXACT, bool LSU>
struct TcConfig {
  static constexpr int kABytes = kBM * kBK * 4;               // 16 KiB
  static constexpr int kBChunkBytes = kBK * 128;              // 32 rows x 32 columns
  static constexpr int kBBytes = (BN / 32) * kBChunkBytes;    // BN / 32 chunks
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kLoOffset = STAGES * kStageBytes;      // sibling lo tiles (3xTF32)
  static constexpr int kTileBytes = (EXACT ? 2 : 1) * STAGES * kStageBytes;
  static constexpr int kProdWarps = LSU ? 4 : 1;
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kEpiWarp0 = kMmaWarp + 1;
  static constexpr int kXformWarps = (EXACT && !LSU) ? 4 : 0;
  static constexpr int kXformWarp0 = kEpiWarp0 + 4;
  static constexpr int kThreads = 32 * (kXformWarp0 + kXformWarps);
  static constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
  static constexpr uint32_t kIdesc = idesc_tf32(kBM, BN, /*b_mn_major=*/true);
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512,
                "TMEM allocation must be a power of two");
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
};

template <int STAGES>
struct alignas(8) TcShared {
  uint64_t full[STAGES];   // stage filled (TMA bytes, or LSU producer warps)
  uint64_t ready[STAGES];  // stage split into hi/lo (3xTF32 with TMA)
  uint64_t empty[STAGES];  // stage consumed by the MMAs (tcgen05.commit)
  uint64_t acc_full[2];    // accumulator complete (tcgen05.commit)
  uint64_t acc_empty[2];   // accumulator drained by the epilogue warps
  uint64_t drain;          // all MMAs issued by this CTA have completed
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

// Byte offset of element (row, col4 * 4 bytes) inside a tile whose rows are
// 128 bytes and whose 1024-byte groups of 8 rows carry the 128-byte swizzle:
// 16-byte chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128(uint32_t linear) {
  return linear ^ (((linear >> 7) & 7u) << 4);
}

// Wait with a warp-uniform outcome (all lanes of the warp wait).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const TcParams &p,
                                          volatile int *abort) {
  bool ok = mbar_wait_bounded(bar, parity, p.timeout_ns, abort, &g_tc_status);
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

__device__ __forceinline__ void store_row_chunk(const TcParams &p, int gm, int gn,
                                                const uint32_t (&r)[32]) {
  if (gm >= p.M) return;
  float *dst = p.C + static_cast<long long>(gm) * p.ldc + gn;
  if (p.vec_store && gn + 32 <= p.N) {
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                             __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
      *reinterpret_cast<float4 *>(dst + j) = v;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (gn + j < p.N) dst[j] = __uint_as_float(r[j]);
  }
}

// Stage one value: raw (TF32 mode: the tensor core drops the low 13 bits) or
// the 3xTF32 pair hi = tf32(x), lo = tf32(x - hi).
template <bool EXACT, int LO_OFFSET>
__device__ __forceinline__ void stage_value(uint8_t *tile, uint32_t off, float v) {
  if (EXACT) {
    const float hi = round_tf32(v);
    const float lo = round_tf32(v - hi);
    *reinterpret_cast<float *>(tile + off) = hi;
    *reinterpret_cast<float *>(tile + LO_OFFSET + off) = lo;
  } else {
    *reinterpret_cast<float *>(tile + off) = v;
  }
}

template <int BN, int STAGES, bool EXACT, bool LSU>
__global__ void __launch_bounds__(TcConfig<BN, STAGES, EXACT, LSU>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const TcParams p) {
  using Cfg = TcConfig<BN, STAGES, EXACT, LSU>;
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
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->acc_full[a], 1);
      mbar_init(&sh->acc_empty[a], 4);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_barrier_init();
  }
  if (!LSU && warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(&sh->tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem_base;

  if (!LSU && warp == 0) {
    // ---------------------------------------------------- TMA producer --
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
          uint8_t *a_dst = tiles + stage * Cfg::kStageBytes;
          uint8_t *b_dst = a_dst + Cfg::kABytes;
          mbar_arrive_expect_tx(&sh->full[stage], Cfg::kStageBytes);
          tma_load_2d(a_dst, &tmap_a, &sh->full[stage], kb * kBK, mb * kBM);
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
            tma_load_2d(b_dst + c * Cfg::kBChunkBytes, &tmap_b, &sh->full[stage],
                        nb * BN + c * 32, kb * kBK);
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
    // ---------------------------------------------------- LSU producer --
    uint32_t stage = 0, phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m0 = mb * kBM, n0 = nb * BN;
      bool ok = true;
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        if (!warp_wait(&sh->empty[stage], phase ^ 1, p, abort)) {
          ok = false;
          break;
        }
        uint8_t *a_st = tiles + stage * Cfg::kStageBytes;
        uint8_t *b_st = a_st + Cfg::kABytes;
        const int k0 = kb * kBK;
        {
          // A: warp w stages rows w, w + 4, ..., lane = k within the stage.
          const int gk = k0 + lane;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int gm = m0 + warp + 4 * i;
            v[i] = (gm < p.M && gk < p.K) ? __ldg(p.A + static_cast<long long>(gm) * p.lda + gk)
                                          : 0.0f;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            stage_value<EXACT, Cfg::kLoOffset>(a_st, sw128((warp + 4 * i) * 128 + lane * 4),
                                               v[i]);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          // B: warp w stages k-rows w + 4 i (i in this half), lane = column in a chunk.
          float v[4][BN / 32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kr = warp + 4 * (half * 4 + i);
            const int gk = k0 + kr;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
              const int gn = n0 + c * 32 + lane;
              v[i][c] = (gk < p.K && gn < p.N)
                            ? __ldg(p.B + static_cast<long long>(gk) * p.ldb + gn)
                            : 0.0f;
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kr = warp + 4 * (half * 4 + i);
#pragma unroll
            for (int c = 0; c < BN / 32; ++c)
              stage_value<EXACT, Cfg::kLoOffset>(
                  b_st, c * Cfg::kBChunkBytes + sw128(kr * 128 + lane * 4), v[i][c]);
          }
        }
        fence_proxy_async_smem();
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
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        if (!mbar_wait_bounded(&sh->acc_empty[acc], acc_phase ^ 1, p.timeout_ns, abort,
                               &g_tc_status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + acc * BN;
        for (int kb = 0; kb < p.num_k_blocks; ++kb) {
          uint64_t *in_bar = (EXACT && !LSU) ? &sh->ready[stage] : &sh->full[stage];
          if (!mbar_wait_bounded(in_bar, phase, p.timeout_ns, abort, &g_tc_status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_hi = smem_addr(tiles + stage * Cfg::kStageBytes);
          const uint32_t b_hi = a_hi + Cfg::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            // A is K-major: a k-step of 8 fp32 is 32 bytes along the swizzled row.
            // B is MN-major: a k-step is one 8-row, 1024-byte swizzle atom;
            // 32-column chunks are kBChunkBytes apart (leading byte offset).
            const uint64_t da = smem_desc(a_hi + kk * 32, 16, 1024, kSw128);
            const uint64_t db = smem_desc(b_hi + kk * 1024, Cfg::kBChunkBytes, 1024, kSw128);
            const uint32_t accumulate = (kb | kk) != 0;
            if (EXACT) {
              const uint64_t da_lo =
                  smem_desc(a_hi + Cfg::kLoOffset + kk * 32, 16, 1024, kSw128);
              const uint64_t db_lo =
                  smem_desc(b_hi + Cfg::kLoOffset + kk * 1024, Cfg::kBChunkBytes, 1024, kSw128);
              mma_tf32(d_tmem, da_lo, db, Cfg::kIdesc, accumulate);
              mma_tf32(d_tmem, da, db_lo, Cfg::kIdesc, 1);
              mma_tf32(d_tmem, da, db, Cfg::kIdesc, 1);
            } else {
              mma_tf32(d_tmem, da, db, Cfg::kIdesc, accumulate);
            }
          }
          mma_commit(&sh->empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&sh->acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // Every MMA this thread issued completes before TMEM is released.
      mma_commit(&sh->drain);
      drain_wait(&sh->drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= Cfg::kEpiWarp0 && warp < Cfg::kEpiWarp0 + 4) {
    // --------------------------------------------------------- epilogue --
    const uint32_t quad = warp & 3;  // TMEM lanes this warp may read
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      if (!warp_wait(&sh->acc_full[acc], acc_phase, p, abort)) break;
      tc_fence_after_sync();
      const int gm = mb * kBM + quad * 32 + lane;
      const uint32_t t_row = tmem + ((quad * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        const int gn = nb * BN + c * 32;
        if (gn >= p.N) break;
        uint32_t r[32];
        tmem_load_32cols(t_row + c * 32, r);
        tmem_load_wait();
        store_row_chunk(p, gm, gn, r);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->acc_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  } else if (Cfg::kXformWarps > 0 && warp >= Cfg::kXformWarp0) {
    // ---------------------------------------------- 3xTF32 split (TMA) --
    const int xt = threadIdx.x - Cfg::kXformWarp0 * 32;
    constexpr int kVecs = Cfg::kStageBytes / 16;
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
      for (int kb = 0; kb < p.num_k_blocks; ++kb) {
        if (!warp_wait(&sh->full[stage], phase, p, abort)) {
          ok = false;
          break;
        }
        float4 *raw = reinterpret_cast<float4 *>(tiles + stage * Cfg::kStageBytes);
        float4 *lo = reinterpret_cast<float4 *>(tiles + Cfg::kLoOffset + stage * Cfg::kStageBytes);
#pragma unroll 4
        for (int i = xt; i < kVecs; i += 32 * Cfg::kXformWarps) {
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
    tmem_dealloc(tmem, Cfg::kTmemCols);
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

// Small cache of encoded tensor maps keyed by (address, extents, pitch, box).
struct MapKey {
  const void *ptr;
  uint64_t d0, d1, pitch;
  uint32_t b0, b1;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && pitch == o.pitch && b0 == o.b0 &&
           b1 == o.b1;
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
// b0 x b1 box, 128-byte swizzle and zero fill outside the matrix.
bool get_map(const void *ptr, uint64_t d0, uint64_t d1, uint64_t pitch_bytes, uint32_t b0,
             uint32_t b1, CUtensorMap *out) {
  static MapCache cache;
  const MapKey key{ptr, d0, d1, pitch_bytes, b0, b1};
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
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
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

template <int BN, int STAGES, bool EXACT, bool LSU>
int launch_variant(const GemmArgs &a, int sm_count, cudaStream_t stream) {
  using Cfg = TcConfig<BN, STAGES, EXACT, LSU>;
  auto kernel = tc_gemm_kernel<BN, STAGES, EXACT, LSU>;
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
    if (!get_map(a.A, a.K, a.M, a.lda * 4, kBK, kBM, &map_a)) return kErrLaunch;
    if (!get_map(a.B, a.N, a.K, a.ldb * 4, 32, kBK, &map_b)) return kErrLaunch;
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
  p.num_m_blocks = static_cast<int>((a.M + kBM - 1) / kBM);
  p.num_n_blocks = static_cast<int>((a.N + BN - 1) / BN);
  p.num_tiles = p.num_m_blocks * p.num_n_blocks;
  p.num_k_blocks = static_cast<int>((a.K + kBK - 1) / kBK);
  p.vec_store = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && (a.ldc % 4 == 0);
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
    if (lsu) return launch_variant<256, 2, true, true>(a, sm_count, stream);
    return launch_variant<256, 2, true, false>(a, sm_count, stream);
  }
  if (lsu) return launch_variant<256, 4, false, true>(a, sm_count, stream);
  return launch_variant<256, 4, false, false>(a, sm_count, stream);
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
