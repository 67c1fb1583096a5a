// tc_gemm.cu -- tensor-core fp32 GEMM for sm_103a (tcgen05 + TMEM).
//
// C[M x N] = A[M x K] * B[K x N], all row-major fp32.
//
// Formulation. Each output tile is computed transposed,
//
//     D = C_tile^T  (128 n x 256 m)  =  B_tile^T (128 n x K)  *  A_tile^T (K x 256 m),
//
// with B_tile^T as the MMA's A operand and the A tile (K-major when A is
// stored M x K) as its B operand in shared memory. B_tile^T sits in TMEM
// (lane = n, one 32-bit column per k) where threads write it, or in shared
// memory as an MN-major tile (B stored K x N: the 32-byte-atom swizzle, the
// one MN-major layout kind::tf32 multiplies from) in the one-pass pair
// kernel. The accumulator D lives in TMEM with lane = n and column = m, so
// each epilogue store writes 32 consecutive columns of one row of C (a
// coalesced 128-byte segment).
//
// Kernels (warp-specialised, persistent, one CTA per SM, grouped raster, the
// same work list, epilogue and split-tile sum):
//   tc_pair_kernel        one TF32 pass on CTA pairs (tcgen05 cta_group::2,
//                         M = 256, N = 256): both operands by TMA, in every
//                         layout, straight from shared memory to the MMA.
//   tc_pair_exact_kernel  3xTF32 on CTA pairs: TMA copies; transform warps
//                         write B^T hi/lo into TMEM and split A into hi (in
//                         place) and lo (sibling tile); B_lo*A_hi,
//                         B_hi*A_lo, B_hi*A_hi per k-step (small terms
//                         first), hi = tf32(x), lo = tf32(x - hi).
//   tc_lsu_kernel         either mode on one SM per tile (M = 128, N = 256),
//                         for operands TMA cannot describe: four warps stage
//                         both with plain loads (A into shared memory, B^T
//                         into TMEM, split on the way for 3xTF32).
// Roles: a producer (one TMA thread or four load warps), one MMA-issuing
// thread, four epilogue warps that read D from TMEM and store C with
// row/column guards, and in the 3xTF32 pair kernel eight transform warps.
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
#include <type_traits>
#include <vector>

#include "../../include/gemm_f32.h"
#include "kernels.h"
#include "ptx.cuh"

namespace gemm {

__device__ int g_tc_status;  // first error recorded by any kernel of this unit

namespace {

constexpr int kTM = 256;        // rows of C per tile   (MMA N)
constexpr int kTN = 128;        // columns of C per tile (MMA M = TMEM lanes)
constexpr int kUmmaK = 8;       // K per tcgen05.mma of kind::tf32
constexpr int kGroupM = 8;      // m-blocks per raster group
constexpr int kClusterSplitMax = 4;  // pairs per cluster: 8 CTAs, the portable cluster size
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;    // D: columns [0, 256) (and [256, 512) when double-buffered)
constexpr uint32_t kBtCol = 256;   // B^T stage buffers from column 256 (B stored K x N)

struct TcParams {
  int M, N, K;
  const float *A;
  long long lda;
  const float *B;
  long long ldb;
  float *C;
  long long ldc;
  int num_m_blocks, num_n_blocks, num_k_blocks;
  // Scheduling is in units of cl CTAs (a cluster) and of "unit tiles" of
  // kTM x (cl * kTN): the cl CTAs of a cluster compute the cl adjacent output
  // tiles of one unit tile and share its A tile.
  int cl, num_nu_blocks, num_tiles;
  // Stream-K schedule (see UnitIter): unit tiles [0, dp_tiles) are whole-tile
  // work dealt round-robin; the k-blocks of unit tiles [dp_tiles, num_tiles)
  // are split into contiguous chunks of sk_share k-blocks over clusters
  // [0, sk_ctas).
  int dp_tiles, sk_share, sk_ctas;
  // Partial sums of split tiles: two kTM x kTN fp32 slots per (cluster, rank)
  // -- one for the first and one for the last unit of the cluster's chunk,
  // the only units that can be parts of a split tile.
  float *sk_partials;
  // Split tiles: parts finished so far per (tile, rank), zeroed before launch.
  unsigned *sk_counters;
  float alpha, beta;       // C = alpha * A op(B) + beta * C (beta == 0: C is not read)
  // Pair kernel: the MN-major A (B) tile comes as one copy of four 32-element
  // chunks through a 3-D tensor map (rows a multiple of 32), else as four.
  int a_one_copy, b_one_copy;
  unsigned long long timeout_ns;
  // Failure-detection self-test only: the pair kernels' producer issues no
  // copy after this many k-blocks, so the other roles' bounded waits run out
  // and the abort path runs. -1 (never stop) in every other launch.
  int stall_kb;
  // Pair kernels on problems with fewer unit tiles than CTA pairs: ks > 1
  // pairs of one cluster share each unit tile, pair q of the cluster taking
  // the q-th of ks contiguous k-slices; every CTA writes its partial tile
  // (its own band of rows to shared memory, the rest to its sk_partials slot)
  // and, after a cluster barrier, sums its band over the ks partials
  // (cluster_split_sum). 1 otherwise.
  int ks;
  // 1: each cluster takes its stream-K chunk before its whole tiles, so that
  // the sums of split tiles run in the epilogue while the MMAs go on with
  // whole tiles; 0: whole tiles first.
  int sk_first;
  // Height, in unit tiles, of the raster groups that order the tiles: kGroupM
  // (concurrent clusters share operand tiles in L2), or 1 (plain row-major
  // order) for a streamed launch.
  int group_m;
  // Streamed launch (operands arriving while the kernel runs; null pointers
  // otherwise). Rows of unit tiles go in groups of stream_group, one word
  // each. Before its first copy of A rows of unit-tile row mb a producer
  // waits until stream_a_ready[mb / stream_group] == stream_epoch; before
  // copying a k-block below stream_kb_split, until stream_b_ready[0] ==
  // stream_epoch, and for one at or above it until stream_b_ready[1] ==
  // stream_epoch. The host's copy stream writes these words once the copies
  // they cover have completed. After storing a whole unit tile, each CTA
  // adds 1 to stream_c_done[mb / stream_group], so a group is in C when its
  // counter reaches cl * num_nu_blocks times its rows of unit tiles; a CTA
  // that gives up raises every counter to kStreamRelease, which every
  // target passes, so the host's waits for C always end.
  const unsigned *stream_a_ready, *stream_b_ready;
  unsigned *stream_c_done;
  unsigned stream_epoch;
  int stream_kb_split, stream_group;
  // Extents in elements of A, B, C and the workspace's partial slots and
  // counters, which the checked build's index checks hold every plain
  // access to (checks.cuh).
  long long a_extent, b_extent, c_extent, partial_extent, counter_extent;
};

// One unit of work of a CTA: k-blocks [kb0, kb1) of unit tile `tile`.
// nparts > 1 marks a split tile: this CTA contributes part `part` of
// `nparts`, sk_tile indexes the tile's counters and slot is this part's
// partial-sum slot pair index (see TcParams::sk_partials).
struct WorkUnit {
  int tile, kb0, kb1, sk_tile, part, nparts, slot;
};

// Slot index of part `part` of split unit tile `s` (2 * cluster + 0 for the
// first unit of that cluster's chunk, + 1 for its last).
__host__ __device__ __forceinline__ int split_slot(const TcParams &p, int s, int part) {
  const int first = (s * p.num_k_blocks) / p.sk_share;
  const int c = first + part;
  if (part > 0) return 2 * c;  // later parts start their cluster's chunk
  // The first part is its cluster's first unit if that chunk starts inside
  // this tile, otherwise its last unit.
  return (c * p.sk_share >= s * p.num_k_blocks) ? 2 * c : 2 * c + 1;
}

// tc_lsu_kernel: operands staged by plain loads (any leading dimension, any
// alignment, A in either storage), one SM per output tile 128 n x 256 m.
// BK = K per stage: 32 (A rows of 128 bytes, 128-byte swizzle) or 16 (rows of
// 64 bytes, 64-byte swizzle). Either way a row of the A tile is one swizzle
// span, 8-row groups are the swizzle atom, and a k-step of 8 advances the
// descriptor by 32 bytes along the row.
// OPB = false: B is stored K x N (N contiguous); the producer warps write its
// tile straight into TMEM as B^T (hi and lo for 3xTF32). OPB = true: B is
// stored transposed, N x K (K contiguous), so its tile is staged K-major like
// A's (with its lo tile for 3xTF32) and read by the MMA from shared memory;
// TMEM then holds only accumulators, two of them.
template <int BK, int STAGES, bool EXACT, bool OPB>
struct TcConfig {
  static_assert(BK == 16 || BK == 32, "BK");
  static constexpr bool kBtTmem = !OPB;                          // B^T operand in TMEM
  static constexpr int kRowBytes = BK * 4;                       // one K-major tile row
  static constexpr int kAtomBytes = 8 * kRowBytes;               // 8-row swizzle atom (SBO)
  static constexpr uint32_t kLayout = BK == 32 ? 2u : 4u;        // 128- or 64-byte swizzle
  static constexpr int kABytes = kTM * BK * 4;                   // A tile, K-major, swizzled
  static constexpr int kBBytes = OPB ? BK * kTN * 4 : 0;         // K-major B tile (OPB)
  // 3xTF32 lo tiles follow the hi tiles at kLoOffset, same layout.
  static constexpr int kLoOffset = kABytes + kBBytes;
  static constexpr int kLoBytes = EXACT ? kABytes + kBBytes : 0;
  static constexpr int kStageBytes = kABytes + kBBytes + kLoBytes;
  static constexpr int kBOffset = kABytes;
  static constexpr int kALoOffset = kLoOffset;
  static constexpr int kBLoOffset = kLoOffset + kABytes;         // OPB && EXACT
  static constexpr int kTileBytes = STAGES * kStageBytes;
  static constexpr uint32_t kBtColsPerStage = kBtTmem ? (EXACT ? 2 * BK : BK) : 0;  // hi (+ lo)
  static constexpr int kAccBufs = kBtTmem ? 1 : 2;               // TMEM accumulators
  static constexpr int kProdWarps = 4;
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kEpiWarp0 = kMmaWarp + 1;
  static constexpr int kThreads = 32 * (kEpiWarp0 + 4);
  static constexpr uint32_t kIdesc = idesc_tf32(kTN, kTM);
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kBtTmem ? kBtCol + STAGES * kBtColsPerStage <= kTmemCols
                        : kAccBufs * kTM <= static_cast<int>(kTmemCols),
                "TMEM budget");
};

template <int STAGES>
struct alignas(8) TcShared {
  uint64_t full[STAGES];   // stage loaded (TMA bytes, or the LSU producer warps)
  uint64_t empty[STAGES];  // stage consumed by the MMAs (tcgen05.commit)
  uint64_t acc_full[2];    // accumulator complete (tcgen05.commit)
  uint64_t acc_empty[2];   // accumulator drained by the epilogue warps
  uint64_t drain;          // every MMA of this CTA (pair) has completed
  uint32_t tmem_base;
  int abort;
  int sk_last;             // epilogue: this CTA finished a split tile last
  int fix_tile, fix_nparts, fix_mb, fix_nb;  // final split tile left for all warps to sum
};

// Unit tile t -> (m-block, n-block of this CTA): grouped raster over unit
// tiles, then the CTA's rank within its cluster picks one of the cl output
// tiles of the unit tile.
__device__ __forceinline__ void tile_coords(const TcParams &p, int t, uint32_t rank, int &mb,
                                            int &nb) {
  const int group_tiles = p.group_m * p.num_nu_blocks;
  const int g = t / group_tiles;
  const int first_m = g * p.group_m;
  const int gm = min(p.num_m_blocks - first_m, p.group_m);
  const int r = t - g * group_tiles;
  mb = first_m + r % gm;
  nb = (r / gm) * p.cl + static_cast<int>(rank);
}

// Bounded wait of a streamed launch until the word at `flag` equals `want`:
// the host's copy stream writes it (a stream memory operation, executed by
// the GPU's front end, not by an SM) once the copies before it have
// completed. The acquire load orders those copies' data before the caller's
// later reads, and the proxy fence before its TMA copies of them. On timeout
// the wait records kStatusTimeout and raises the CTA's abort flag.
__device__ __noinline__ bool stream_flag_wait(const unsigned *flag, unsigned want,
                                              unsigned long long timeout_ns,
                                              volatile int *abort) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v == want) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (*abort) return false;
    if (it == 0) {
      t0 = global_timer_ns();
    } else if (global_timer_ns() - t0 > timeout_ns) {
      *abort = 1;
      atomicCAS(&g_tc_status, 0, kStatusTimeout);
      return false;
    }
    __nanosleep(256);
  }
}

// A producer's waits in a streamed launch (TcParams::stream_*): the row of
// unit tiles of A before a tile's copies, each half of B's k range before
// its first k-block. Nothing to wait for in any other launch.
struct StreamGate {
  bool b_have[2] = {false, false};
  __device__ __forceinline__ bool tile(const TcParams &p, int mb, volatile int *abort) {
    return p.stream_a_ready == nullptr ||
           stream_flag_wait(&p.stream_a_ready[mb / p.stream_group], p.stream_epoch, p.timeout_ns,
                            abort);
  }
  __device__ __forceinline__ bool kblock(const TcParams &p, int kb, volatile int *abort) {
    if (p.stream_b_ready == nullptr) return true;
    const int h = kb < p.stream_kb_split ? 0 : 1;
    if (!b_have[h])
      b_have[h] = stream_flag_wait(&p.stream_b_ready[h], p.stream_epoch, p.timeout_ns, abort);
    return b_have[h];
  }
};

// A streamed launch whose CTA gave up: raise every done counter to
// kStreamRelease, so that the host's copies of C (waiting on the counters)
// go ahead and the call returns the recorded error.
__device__ __forceinline__ void stream_release(const TcParams &p, bool aborted) {
  if (p.stream_c_done == nullptr || !aborted || threadIdx.x != 0) return;
  const int words = (p.num_m_blocks + p.stream_group - 1) / p.stream_group;
  for (int r = 0; r < words; ++r) atomicMax(&p.stream_c_done[r], kStreamRelease);
}

// The work list of one cluster c (both CTAs of a cluster walk the same list),
// identical for every role: the whole unit tiles c, c + clusters, ... below
// dp_tiles (raster order, so concurrent clusters share operand tiles in L2)
// and its stream-K chunk (k-blocks [c * share, (c + 1) * share) of the
// remaining unit tiles, in order, cut at tile boundaries): whole tiles first,
// or with TcParams::sk_first the chunk first. Every cluster sees
// the same partition, so the number of clusters contributing to a split tile
// and each one's part index follow from the chunk boundaries alone.
// (Host and device code: the host-side self-check gemm_f32_schedule_check
// walks the same work lists.)
__host__ __device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

struct UnitIter {
  int sk_pos, sk_end, dp_next;
  int c, workers;
  // The work list of cluster `cluster` of `clusters`.
  __host__ __device__ UnitIter(const TcParams &p, int cluster, int clusters) {
    c = cluster;
    workers = clusters;
    const int sk_total = (p.num_tiles - p.dp_tiles) * p.num_k_blocks;
    if (c < p.sk_ctas && sk_total > 0) {
      sk_pos = imin(c * p.sk_share, sk_total);
      sk_end = imin(sk_pos + p.sk_share, sk_total);
    } else {
      sk_pos = sk_end = 0;
    }
    dp_next = c;
  }
  // This CTA's cluster.
  __device__ explicit UnitIter(const TcParams &p)
      : UnitIter(p, static_cast<int>(blockIdx.x) / p.cl, static_cast<int>(gridDim.x) / p.cl) {}
  __host__ __device__ bool next(const TcParams &p, WorkUnit &u) {
    if (p.ks > 1) {
      // One k-slice of one unit tile: pair c takes slice c % ks of tile c / ks.
      if (dp_next < 0) return false;
      const int q = c % p.ks;
      u.tile = c / p.ks;
      u.kb0 = (q * p.num_k_blocks) / p.ks;
      u.kb1 = ((q + 1) * p.num_k_blocks) / p.ks;
      u.sk_tile = -1;
      u.part = q;
      u.nparts = p.ks;
      u.slot = -1;
      dp_next = -1;
      return true;
    }
    if (p.sk_first) return next_split(p, u) || next_whole(p, u);
    return next_whole(p, u) || next_split(p, u);
  }
  __host__ __device__ bool next_whole(const TcParams &p, WorkUnit &u) {
    if (dp_next < p.dp_tiles) {
      u.tile = dp_next;
      u.kb0 = 0;
      u.kb1 = p.num_k_blocks;
      u.sk_tile = -1;
      u.part = 0;
      u.nparts = 1;
      u.slot = -1;
      dp_next += workers;
      return true;
    }
    return false;
  }
  __host__ __device__ bool next_split(const TcParams &p, WorkUnit &u) {
    if (sk_pos < sk_end) {
      const int kbt = p.num_k_blocks;
      const int s = sk_pos / kbt;
      u.sk_tile = s;
      u.tile = p.dp_tiles + s;
      u.kb0 = sk_pos - s * kbt;
      u.kb1 = imin(kbt, u.kb0 + (sk_end - sk_pos));
      const int first = (s * kbt) / p.sk_share;
      const int last = ((s + 1) * kbt - 1) / p.sk_share;
      u.nparts = last - first + 1;
      u.part = c - first;
      u.slot = split_slot(p, s, u.part);
      sk_pos += u.kb1 - u.kb0;
      return true;
    }
    return false;
  }
  // True when no unit follows the one last returned by next().
  __host__ __device__ bool done(const TcParams &p) const {
    if (p.ks > 1) return dp_next < 0;
    return dp_next >= p.dp_tiles && sk_pos >= sk_end;
  }
};

// alpha * acc + beta * C (C read only when beta != 0).
__device__ __forceinline__ float scale_out(const TcParams &p, float acc, const float *c) {
  const float v = p.alpha * acc;
  return p.beta != 0.0f ? v + p.beta * *c : v;
}

// The same with C's element already loaded (c is not used when beta == 0).
__device__ __forceinline__ float scale_value(const TcParams &p, float acc, float c) {
  const float v = p.alpha * acc;
  return p.beta != 0.0f ? v + p.beta * c : v;
}

// Sum the partial tiles of split tile `sk_tile` in part order and store the
// result to C. Run by `nthreads` threads of the CTA that finished last: the
// four epilogue warps, or every warp of the CTA for its final unit. The tile
// is read as float4s, BATCH per thread and part in flight at a time (the sum
// is bound by how many loads are in flight, not by bandwidth).
template <int BATCH = 8>
__device__ __forceinline__ void epilogue_fixup(const TcParams &p, int sk_tile, uint32_t rank,
                                            int nparts, int mb, int nb, int tid, int nthreads) {
  constexpr int kVec = kTM * kTN / 4;  // float4s per tile
  constexpr int kRowVec = kTN / 4;     // float4s per tile row
  constexpr int kBatch = BATCH;
  const long long slot4 = static_cast<long long>(kTM) * kTN / 4;
  // Slot (index, rank) starts at (index * cl + rank) * slot4 float4s.
  const float4 *parts = reinterpret_cast<const float4 *>(p.sk_partials) + rank * slot4;
  const float4 *base = parts + static_cast<long long>(split_slot(p, sk_tile, 0)) * p.cl * slot4;
  // Scalars of p in registers: the stores to C could otherwise alias p and
  // force reloads.
  const int M = p.M, N = p.N;
  const long long ldc = p.ldc;
  float *__restrict__ const C = p.C;
  const float alpha = p.alpha, beta = p.beta;
  const bool vec_ok = (ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(C) % 16 == 0);
#pragma unroll 1
  for (int f0 = 0; f0 < kVec; f0 += nthreads * kBatch) {
    float4 acc[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int f = f0 + tid + nthreads * j;
      acc[j] = f < kVec && ptr_ok(kSitePartialRead, base + f, 4, p.sk_partials, p.partial_extent)
                   ? __ldcg(base + f)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll 1
    for (int q = 1; q < nparts; ++q) {
      const float4 *src = parts + static_cast<long long>(split_slot(p, sk_tile, q)) * p.cl * slot4;
      float4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int f = f0 + tid + nthreads * j;
        v[j] = f < kVec && ptr_ok(kSitePartialRead, src + f, 4, p.sk_partials, p.partial_extent)
                   ? __ldcg(src + f)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        acc[j].x += v[j].x;
        acc[j].y += v[j].y;
        acc[j].z += v[j].z;
        acc[j].w += v[j].w;
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int f = f0 + tid + nthreads * j;
      if (f >= kVec) continue;
      const int gm = mb * kTM + f / kRowVec;
      const int gn = nb * kTN + (f % kRowVec) * 4;
      if (gm >= M) continue;
      float *dst = C + static_cast<long long>(gm) * ldc + gn;
      if (vec_ok && gn + 3 < N) {
        if (!ptr_ok(kSiteCStore, dst, 4, C, p.c_extent)) continue;
        float4 v = make_float4(alpha * acc[j].x, alpha * acc[j].y, alpha * acc[j].z,
                               alpha * acc[j].w);
        if (beta != 0.0f) {
          const float4 c = *reinterpret_cast<const float4 *>(dst);
          v.x += beta * c.x;
          v.y += beta * c.y;
          v.z += beta * c.z;
          v.w += beta * c.w;
        }
        *reinterpret_cast<float4 *>(dst) = v;
      } else {
        const float e[4] = {acc[j].x, acc[j].y, acc[j].z, acc[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (gn + i < N && ptr_ok(kSiteCStore, dst + i, 1, C, p.c_extent))
            dst[i] = beta != 0.0f ? alpha * e[i] + beta * dst[i] : alpha * e[i];
      }
    }
  }
}

// float4s per thread and partial in flight in cluster_split_sum.
constexpr int kClusterSumBatch = 8;

// Rows [row0, row1) of the kTM-row tile that pair q of ks sums in a cluster
// split (the band the CTAs of that pair own).
__device__ __forceinline__ void cluster_split_band(int ks, int q, int &row0, int &row1) {
  row0 = (q * kTM) / ks;
  row1 = ((q + 1) * kTM) / ks;
}

// The final sum of a cluster-split tile (TcParams::ks > 1), run by all
// nthreads threads of every CTA once each CTA of the cluster has written its
// k-slice partial ([m][n], kTN floats per row) and a cluster barrier has
// ordered those writes: the rows of its own band in its shared memory at
// own, the other rows in its slot of sk_partials (slot = CTA index). The
// CTAs of rank r (0, 1) in the ks pairs hold the same 128 n x 256 m output
// tile; pair q's CTA sums its band of rows over the ks partials, added in
// pair order 0 .. ks-1 (so results do not depend on timing), scales by alpha,
// adds beta C and stores C with row and column guards. The other pairs'
// partials were written by other SMs, so they are read through L2
// (ld.global.cg), BATCH float4s per thread and partial in flight.
template <int BATCH>
__device__ __forceinline__ void cluster_split_sum(const TcParams &p, const float *own,
                                                  uint32_t crank, int tid, int nthreads) {
  const int ks = p.ks;
  const uint32_t r = crank & 1u, q = crank >> 1;
  int mb, nb;
  tile_coords(p, (static_cast<int>(blockIdx.x) >> 1) / ks, r, mb, nb);
  int row0, row1;
  cluster_split_band(ks, static_cast<int>(q), row0, row1);
  constexpr int kRowVec = kTN / 4;
  constexpr long long kSlotVec = static_cast<long long>(kTM) * kTN / 4;
  const float4 *own4 = reinterpret_cast<const float4 *>(own) + row0 * kRowVec;
  const int nvec = (row1 - row0) * kRowVec;
  // Slot of the CTA of rank r in pair 0 of this cluster; pair j's is 2 j further.
  const float4 *base = reinterpret_cast<const float4 *>(p.sk_partials) +
                       (static_cast<long long>(blockIdx.x) - crank + r) * kSlotVec +
                       static_cast<long long>(row0) * kRowVec;
  const int M = p.M, N = p.N;
  const long long ldc = p.ldc;
  float *__restrict__ const C = p.C;
  const float alpha = p.alpha, beta = p.beta;
  const bool vec_ok = (ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(C) % 16 == 0);
#pragma unroll 1
  for (int f0 = tid; f0 < nvec; f0 += nthreads * BATCH) {
    float4 acc[BATCH];
#pragma unroll
    for (int j = 0; j < kClusterSplitMax; ++j) {
      if (j >= ks) break;
      float4 v[BATCH];
      if (static_cast<uint32_t>(j) == q) {
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
          const int f = f0 + b * nthreads;
          v[b] = f < nvec && index_ok(kSiteBand, (row0 * kRowVec + f) * 4LL, 4, kTM * kTN)
                     ? own4[f]
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      } else {
        const float4 *src = base + 2 * j * kSlotVec;
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
          const int f = f0 + b * nthreads;
          v[b] = f < nvec && ptr_ok(kSitePartialRead, src + f, 4, p.sk_partials, p.partial_extent)
                     ? __ldcg(src + f)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int b = 0; b < BATCH; ++b) {
        if (j == 0) {
          acc[b] = v[b];
        } else {
          acc[b].x += v[b].x;
          acc[b].y += v[b].y;
          acc[b].z += v[b].z;
          acc[b].w += v[b].w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int f = f0 + b * nthreads;
      if (f >= nvec) continue;
      const int gm = mb * kTM + row0 + f / kRowVec, gn = nb * kTN + (f % kRowVec) * 4;
      if (gm >= M) continue;
      float *dst = C + static_cast<long long>(gm) * ldc + gn;
      if (vec_ok && gn + 3 < N) {
        if (!ptr_ok(kSiteCStore, dst, 4, C, p.c_extent)) continue;
        float4 o = make_float4(alpha * acc[b].x, alpha * acc[b].y, alpha * acc[b].z,
                               alpha * acc[b].w);
        if (beta != 0.0f) {
          const float4 c = *reinterpret_cast<const float4 *>(dst);
          o.x += beta * c.x;
          o.y += beta * c.y;
          o.z += beta * c.z;
          o.w += beta * c.w;
        }
        *reinterpret_cast<float4 *>(dst) = o;
      } else {
        const float e[4] = {acc[b].x, acc[b].y, acc[b].z, acc[b].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (gn + i < N && ptr_ok(kSiteCStore, dst + i, 1, C, p.c_extent))
            dst[i] = beta != 0.0f ? alpha * e[i] + beta * dst[i] : alpha * e[i];
      }
    }
  }
}

// Swizzled byte offset of a linear offset inside an A tile whose rows are
// BK * 4 bytes: the 16-byte chunk index within a row is XORed with address
// bits 7.. (row mod 8 for 128-byte rows, (row / 2) mod 4 for 64-byte rows),
// the pattern the TMA unit writes and the MMA descriptor expects.
template <int BK>
__device__ __forceinline__ uint32_t swizzle_a(uint32_t linear) {
  return BK == 32 ? linear ^ (((linear >> 7) & 7u) << 4) : linear ^ (((linear >> 7) & 3u) << 4);
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

template <int W>
__device__ __forceinline__ void tmem_store_row(uint32_t taddr, const uint32_t (&r)[W]) {
  if constexpr (W == 32)
    tmem_store_32cols(taddr, r);
  else if constexpr (W == 16)
    tmem_store_16cols(taddr, r);
  else if constexpr (W == 8)
    tmem_store_8cols(taddr, r);
  else
    tmem_store_4cols(taddr, r);
}

// W values of B^T row n (part of the stage's k range) into TMEM, raw or as
// the 3xTF32 pair hi = tf32(x), lo = tf32(x - hi).
template <int W, bool EXACT>
__device__ __forceinline__ void bt_to_tmem(uint32_t t_hi, uint32_t t_lo, const float (&v)[W]) {
  uint32_t hi[W];
  if (EXACT) {
    uint32_t lo[W];
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float h = round_tf32(v[k]);
      hi[k] = __float_as_uint(h);
      lo[k] = __float_as_uint(round_tf32(v[k] - h));
    }
    tmem_store_row<W>(t_hi, hi);
    tmem_store_row<W>(t_lo, lo);
  } else {
#pragma unroll
    for (int k = 0; k < W; ++k) hi[k] = __float_as_uint(v[k]);
    tmem_store_row<W>(t_hi, hi);
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

// Plain-load staging of `rows` rows (r0 + row, row < rows) x BK k (k0 + k) of
// a row-major matrix with leading dimension ld into a K-major swizzled tile
// (zero outside [0, limit_r) x [0, K)); with EXACT the hi part goes to the
// tile and the lo part lo_offset bytes further. Four producer warps, warp w
// taking rows w * (32 / BK) + ..., one BK-wide row segment per 32 / BK lanes.
template <int BK, bool EXACT, int ROWS>
__device__ __forceinline__ void stage_rows_lsu(uint8_t *tile, int lo_offset, const float *src,
                                               long long ld, int r0, int limit_r, int k0, int K,
                                               uint32_t warp, uint32_t lane, int row_bytes,
                                               int site, long long extent) {
  constexpr int kRowsPerInstr = 32 / BK;
  constexpr int kSteps = ROWS / (4 * kRowsPerInstr);
  constexpr int kChunk = kSteps < 32 ? kSteps : 32;  // loads in flight per lane
  static_assert(kSteps % kChunk == 0, "rows per producer pass");
  const int k_in = lane % BK;
  const int r_in = lane / BK;
  const int gk = k0 + k_in;
#pragma unroll 1
  for (int chunk = 0; chunk < kSteps / kChunk; ++chunk) {
    float v[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int row = (chunk * kChunk + i) * 4 * kRowsPerInstr + warp * kRowsPerInstr + r_in;
      const int gr = r0 + row;
      const long long off = static_cast<long long>(gr) * ld + gk;
      v[i] = (gr < limit_r && gk < K && index_ok(site, off, 1, extent)) ? __ldg(src + off) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int row = (chunk * kChunk + i) * 4 * kRowsPerInstr + warp * kRowsPerInstr + r_in;
      stage_a_value<EXACT>(tile, lo_offset, swizzle_a<BK>(row * row_bytes + k_in * 4), v[i]);
    }
  }
}

// Plain-load staging of the same tile from a matrix stored transposed: element
// (row r, k) at src[k * ld + r] (rows contiguous). Lane l covers rows
// 8g + l % 8 and k 4h + l / 8 of an 8 x 4 block, so one load instruction
// reads four fully used 32-byte segments and one store instruction hits 32
// distinct banks of the swizzled tile (eight rows give eight distinct XOR
// patterns, four k the four words of a 16-byte chunk). Four producer warps
// take the blocks in turn.
template <int BK, bool EXACT, int ROWS>
__device__ __forceinline__ void stage_cols_lsu(uint8_t *tile, int lo_offset, const float *src,
                                               long long ld, int r0, int limit_r, int k0, int K,
                                               uint32_t warp, uint32_t lane, int row_bytes,
                                               int site, long long extent) {
  constexpr int kRowGroups = ROWS / 8;
  constexpr int kPerWarp = kRowGroups * (BK / 4) / 4;
  constexpr int kChunk = kPerWarp < 16 ? kPerWarp : 16;  // loads in flight per lane
  static_assert(kPerWarp % kChunk == 0, "blocks per producer pass");
  const int r_in = static_cast<int>(lane & 7u);
  const int k_in = static_cast<int>(lane >> 3);
#pragma unroll 1
  for (int chunk = 0; chunk < kPerWarp / kChunk; ++chunk) {
    float v[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int g = (chunk * kChunk + i) * 4 + static_cast<int>(warp);
      const int row = (g % kRowGroups) * 8 + r_in;
      const int k = (g / kRowGroups) * 4 + k_in;
      const int gr = r0 + row, gk = k0 + k;
      const long long off = static_cast<long long>(gk) * ld + gr;
      v[i] = (gr < limit_r && gk < K && index_ok(site, off, 1, extent)) ? __ldg(src + off) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int g = (chunk * kChunk + i) * 4 + static_cast<int>(warp);
      const int row = (g % kRowGroups) * 8 + r_in;
      const int k = (g / kRowGroups) * 4 + k_in;
      stage_a_value<EXACT>(tile, lo_offset, swizzle_a<BK>(row * row_bytes + k * 4), v[i]);
    }
  }
}

// Epilogue role: four warps (EPI_WARP0 ..) take each finished accumulator
// of the CTA's work list out of TMEM (lane = n, column = m) and either store
// it to C or, for a part of a split tile, to its partial-sum slot; the last
// part to finish sums all parts in order. PAIR: the accumulator's empty
// barrier belongs to the even CTA of the pair (cluster rank pb), which issues
// the MMAs of both. CS (cluster split): the CTA's one accumulator is a k-slice
// of a tile shared by the pairs of its cluster; its rows go ([m][n], kTN
// floats per row) to this CTA's shared memory at own_smem if they are in the
// band this CTA sums, else to its slot of sk_partials, for cluster_split_sum.
template <int ACC_BUFS, int EPI_WARP0, bool PAIR, bool CS = false, bool SCALED = true,
          class Shared>
__device__ __forceinline__ void epilogue_role(const TcParams &p, Shared *sh, uint32_t tmem,
                                              uint32_t warp, uint32_t lane, uint32_t rank,
                                              volatile int *abort, uint32_t pb = 0,
                                              float *own_smem = nullptr) {
  auto release_acc = [pb](uint64_t *bar) {
    if (PAIR)
      mbar_arrive_cluster(bar, pb);
    else
      mbar_arrive(bar);
  };
  const uint32_t quad = warp & 3;  // TMEM lanes (columns of C) this warp may read
  uint32_t acc = 0, acc_phase = 0;
  UnitIter it(p);
  WorkUnit u;
  while (it.next(p, u)) {
    int mb, nb;
    tile_coords(p, u.tile, rank, mb, nb);
    // The four epilogue warps continue or give up together: the split-tile
    // path below synchronises them with named barriers.
    if (!named_barrier_and(1, 128, warp_wait(&sh->acc_full[acc], acc_phase, p, abort))) break;
    tc_fence_after_sync();
    const int n_loc = quad * 32 + lane;
    const int gn = nb * kTN + n_loc;
    const bool n_ok = gn < p.N;
    const uint32_t t_lane = tmem + ((quad * 32) << 16) + kAccCol + acc * kTM;
    if constexpr (CS) {
      float *slot = p.sk_partials + static_cast<long long>(blockIdx.x) * kTM * kTN + n_loc;
      float *local = own_smem + n_loc;
      int row0, row1;
      cluster_split_band(p.ks, u.part, row0, row1);
      auto put = [&](int m, uint32_t v) {
        if (m >= row0 && m < row1) {
          if (index_ok(kSiteBand, m * kTN + n_loc, 1, kTM * kTN))
            local[m * kTN] = __uint_as_float(v);
        } else if (ptr_ok(kSitePartialWrite, slot + m * kTN, 1, p.sk_partials,
                          p.partial_extent)) {
          slot[m * kTN] = __uint_as_float(v);
        }
      };
#pragma unroll 1
      for (int c = 0; c < kTM / 32; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_load_32cols(t_lane + c * 32, r0);
        tmem_load_32cols(t_lane + (c + 1) * 32, r1);
        tmem_load_wait();
        tmem_regs_ready(r0);
        tmem_regs_ready(r1);
#pragma unroll
        for (int j = 0; j < 32; ++j) put(c * 32 + j, r0[j]);
#pragma unroll
        for (int j = 0; j < 32; ++j) put(c * 32 + 32 + j, r1[j]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) release_acc(&sh->acc_empty[acc]);
    } else if (u.nparts == 1) {
      if constexpr (!SCALED) {
        // Whole tile: straight to C, two 32-column chunks per TMEM load wait.
        auto store_chunk = [&](int c, const uint32_t (&r)[32]) {
          const int gm0 = mb * kTM + c * 32;
          if (gm0 >= p.M || !n_ok) return;
          float *dst = p.C + static_cast<long long>(gm0) * p.ldc + gn;
          const int rows = min(32, p.M - gm0);
          // Index checks (checked build): each element's offset in C.
          auto c_ok = [&](int j) {
            return ptr_ok(kSiteCStore, dst + static_cast<long long>(j) * p.ldc, 1, p.C, p.c_extent);
          };
          if (p.alpha == 1.0f && p.beta == 0.0f) {
            if (rows == 32) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c_ok(j)) dst[static_cast<long long>(j) * p.ldc] = __uint_as_float(r[j]);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < rows && c_ok(j)) dst[static_cast<long long>(j) * p.ldc] = __uint_as_float(r[j]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < rows && c_ok(j)) {
                float *d = dst + static_cast<long long>(j) * p.ldc;
                *d = scale_out(p, __uint_as_float(r[j]), d);
              }
          }
        };
#pragma unroll 1
        for (int c = 0; c < kTM / 32; c += 2) {
          if (mb * kTM + c * 32 >= p.M) break;
          uint32_t r0[32], r1[32];
          tmem_load_32cols(t_lane + c * 32, r0);
          tmem_load_32cols(t_lane + (c + 1) * 32, r1);
          tmem_load_wait();
          tmem_regs_ready(r0);
          tmem_regs_ready(r1);
          store_chunk(c, r0);
          store_chunk(c + 1, r1);
        }
      } else {
        auto c_ok = [&](const float *d) {  // index check (checked build)
          return ptr_ok(kSiteCStore, d, 1, p.C, p.c_extent);
        };
        // alpha * acc + beta * C, one 32-column chunk at a time: its 32
        // elements of C are loaded first, all in flight together and under
        // the TMEM load, then scaled and stored (with beta = 0 nothing is
        // loaded). A load right after each store, which the compiler cannot
        // move ahead of it (the addresses differ by an ldc it cannot see is
        // non-zero), waited out a memory round trip per element. The pair
        // kernels hold this code only in their build for alpha != 1 or
        // beta != 0 (in the other it cost registers and 2.5 % at beta = 0);
        // the plain-load kernel, built once, takes it for every call.
        if (p.beta != 0.0f && n_ok) {
          // The whole tile's C into L2 first (the warp's 32 columns are one
          // 128-byte line per row; lanes take every 32nd row), so that only
          // the first chunk's loads wait on HBM.
          const float *col = p.C + static_cast<long long>(mb) * kTM * p.ldc + gn;
#pragma unroll 1
          for (int m = lane; m < kTM && mb * kTM + m < p.M; m += 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(col + static_cast<long long>(m) * p.ldc));
        }
#pragma unroll 1
        for (int c = 0; c < kTM / 32; ++c) {
          const int gm0 = mb * kTM + c * 32;
          if (gm0 >= p.M) break;
          const int rows = n_ok ? min(32, p.M - gm0) : 0;
          float *dst = p.C + static_cast<long long>(gm0) * p.ldc + gn;
          uint32_t r[32];
          tmem_load_32cols(t_lane + c * 32, r);
#pragma unroll
          for (int j0 = 0; j0 < 32; j0 += 16) {
            float cv[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float *d = dst + static_cast<long long>(j0 + j) * p.ldc;
              cv[j] = (p.beta != 0.0f && j0 + j < rows && c_ok(d)) ? *d : 0.0f;
            }
            if (j0 == 0) {
              tmem_load_wait();
              tmem_regs_ready(r);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float *d = dst + static_cast<long long>(j0 + j) * p.ldc;
              if (j0 + j < rows && c_ok(d)) *d = scale_value(p, __uint_as_float(r[j0 + j]), cv[j]);
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) release_acc(&sh->acc_empty[acc]);
      if (p.stream_c_done != nullptr) {
        // Streamed launch: count the tile once the four warps' stores are
        // visible to the host's copy of C.
        __threadfence();
        named_barrier_sync(1, 128);
        if (warp == EPI_WARP0 && lane == 0) atomicAdd(&p.stream_c_done[mb / p.stream_group], 1u);
      }
    } else {
      // Split tile: write this part's partial sums ([m][n], pitch kTN) to
      // its slot and free the accumulator; the last part to finish sums all
      // parts in part order (a fixed order, so results are deterministic)
      // and writes C.
      const long long slot_elems = static_cast<long long>(kTM) * kTN;
      float *slot =
          p.sk_partials + (static_cast<long long>(u.slot) * p.cl + rank) * slot_elems;
#pragma unroll 1
      for (int c = 0; c < kTM / 32; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_load_32cols(t_lane + c * 32, r0);
        tmem_load_32cols(t_lane + (c + 1) * 32, r1);
        tmem_load_wait();
        tmem_regs_ready(r0);
        tmem_regs_ready(r1);
        float *dst = slot + (c * 32) * kTN + n_loc;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (ptr_ok(kSitePartialWrite, dst + j * kTN, 1, p.sk_partials, p.partial_extent))
            dst[j * kTN] = __uint_as_float(r0[j]);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (ptr_ok(kSitePartialWrite, dst + (32 + j) * kTN, 1, p.sk_partials, p.partial_extent))
            dst[(32 + j) * kTN] = __uint_as_float(r1[j]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) release_acc(&sh->acc_empty[acc]);
      __threadfence();
      named_barrier_sync(1, 128);
      if (warp == EPI_WARP0 && lane == 0) {
        const long long ci = static_cast<long long>(u.sk_tile) * p.cl + rank;
        sh->sk_last = index_ok(kSiteCounter, ci, 1, p.counter_extent) &&
                      atomicAdd(&p.sk_counters[ci], 1u) == static_cast<unsigned>(u.nparts - 1);
      }
      named_barrier_sync(1, 128);
      if (sh->sk_last) {
        if (it.done(p)) {
          // The CTA's final unit: every warp sums it after the role loops.
          if (warp == EPI_WARP0 && lane == 0) {
            sh->fix_tile = u.sk_tile;
            sh->fix_nparts = u.nparts;
            sh->fix_mb = mb;
            sh->fix_nb = nb;
          }
        } else {
          __threadfence();
          epilogue_fixup(p, u.sk_tile, rank, u.nparts, mb, nb, threadIdx.x - EPI_WARP0 * 32,
                         128);
        }
      }
      named_barrier_sync(1, 128);  // sk_last is reused by the next split tile
    }
    if (++acc == ACC_BUFS) {
      acc = 0;
      acc_phase ^= 1;
    }
  }
}

// The tensor maps are unused: the parameter list is that of the TMA-fed
// kernels, so one launch path serves all of them.
template <int BK, int STAGES, bool EXACT, bool OPB, bool OPA>
__global__ void __launch_bounds__(TcConfig<BK, STAGES, EXACT, OPB>::kThreads, 1)
    tc_lsu_kernel(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                  const TcParams p) {
  using Cfg = TcConfig<BK, STAGES, EXACT, OPB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcShared<STAGES> *sh = reinterpret_cast<TcShared<STAGES> *>(tiles + Cfg::kTileBytes);
  volatile int *abort = &sh->abort;

  const uint32_t warp = warp_index();
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t rank = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full[s], Cfg::kProdWarps);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->acc_full[a], 1);
      mbar_init(&sh->acc_empty[a], 4);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    sh->fix_tile = -1;
    fence_barrier_init();
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  grid_dependency_wait();  // see tc_pair_kernel

  if (warp < Cfg::kProdWarps) {
    // ---------------------------------------------------------- producer --
    // Warp w stages A rows w, w + 4, ... (lane = k) and B^T rows
    // n = 32 w + lane (TMEM lanes of this warp's quadrant).
    uint32_t stage = 0, phase = 0;
    const uint32_t quad = warp & 3;
    UnitIter it(p);
    WorkUnit u;
    while (it.next(p, u)) {
      int mb, nb;
      tile_coords(p, u.tile, rank, mb, nb);
      const int m0 = mb * kTM, n0 = nb * kTN;
      bool ok = true;
      for (int kb = u.kb0; kb < u.kb1; ++kb) {
        if (!warp_wait(&sh->empty[stage], phase ^ 1, p, abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint8_t *st = tiles + stage * Cfg::kStageBytes;
        const int k0 = kb * BK;
        if (OPA)
          stage_cols_lsu<BK, EXACT, kTM>(st, Cfg::kALoOffset, p.A, p.lda, m0, p.M, k0, p.K, warp,
                                         lane, Cfg::kRowBytes, kSiteLoadA, p.a_extent);
        else
          stage_rows_lsu<BK, EXACT, kTM>(st, Cfg::kALoOffset, p.A, p.lda, m0, p.M, k0, p.K, warp,
                                         lane, Cfg::kRowBytes, kSiteLoadA, p.a_extent);
        if (OPB) {
          // B stored N x K: its tile is staged K-major, like A's.
          stage_rows_lsu<BK, EXACT, kTN>(st + Cfg::kBOffset, Cfg::kBLoOffset - Cfg::kBOffset, p.B,
                                         p.ldb, n0, p.N, k0, p.K, warp, lane, Cfg::kRowBytes,
                                         kSiteLoadB, p.b_extent);
        } else {
          const int gn = n0 + quad * 32 + lane;
          float v[BK];
#pragma unroll
          for (int k = 0; k < BK; ++k) {
            const long long off = static_cast<long long>(k0 + k) * p.ldb + gn;
            v[k] = (gn < p.N && k0 + k < p.K && index_ok(kSiteLoadB, off, 1, p.b_extent))
                       ? __ldg(p.B + off)
                       : 0.0f;
          }
          const uint32_t col = tmem + ((quad * 32) << 16) + kBtCol + stage * Cfg::kBtColsPerStage;
          bt_to_tmem<BK, EXACT>(col, col + BK, v);
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
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      UnitIter it(p);
      WorkUnit u;
      while (ok && it.next(p, u)) {
        if (!mbar_wait_bounded(&sh->acc_empty[acc], acc_phase ^ 1, p.timeout_ns, abort,
                               &g_tc_status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + kAccCol + acc * kTM;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&sh->full[stage], phase, p.timeout_ns, abort, &g_tc_status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_hi = smem_addr(tiles + stage * Cfg::kStageBytes);
          const uint32_t bt_hi = tmem + kBtCol + stage * Cfg::kBtColsPerStage;
#pragma unroll
          for (int kk = 0; kk < BK / kUmmaK; ++kk) {
            // A tile, K-major: a k-step of 8 fp32 is 32 bytes along the swizzled row;
            // 8-row groups (the swizzle atom) are kAtomBytes apart.
            const uint64_t da = smem_desc(a_hi + kk * 32, 16, Cfg::kAtomBytes, Cfg::kLayout);
            const uint32_t accumulate = (kb != u.kb0 || kk != 0) ? 1u : 0u;
            if constexpr (OPB) {
              // B^T rows straight from the K-major B tile in shared memory.
              const uint64_t db = smem_desc(a_hi + Cfg::kBOffset + kk * 32, 16, Cfg::kAtomBytes,
                                            Cfg::kLayout);
              if (EXACT) {
                const uint64_t da_lo = smem_desc(a_hi + Cfg::kALoOffset + kk * 32, 16,
                                                 Cfg::kAtomBytes, Cfg::kLayout);
                const uint64_t db_lo = smem_desc(a_hi + Cfg::kBLoOffset + kk * 32, 16,
                                                 Cfg::kAtomBytes, Cfg::kLayout);
                mma_tf32(d_tmem, db_lo, da, Cfg::kIdesc, accumulate);
                mma_tf32(d_tmem, db, da_lo, Cfg::kIdesc, 1);
                mma_tf32(d_tmem, db, da, Cfg::kIdesc, 1);
              } else {
                mma_tf32(d_tmem, db, da, Cfg::kIdesc, accumulate);
              }
            } else if (EXACT) {
              const uint64_t da_lo =
                  smem_desc(a_hi + Cfg::kALoOffset + kk * 32, 16, Cfg::kAtomBytes, Cfg::kLayout);
              mma_tf32_ts(d_tmem, bt_hi + BK + kk * kUmmaK, da, Cfg::kIdesc, accumulate);
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
        mma_commit(&sh->acc_full[acc]);
        if (++acc == Cfg::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // Every MMA this thread issued completes before TMEM is released.
      mma_commit(&sh->drain);
      drain_wait(&sh->drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    epilogue_role<Cfg::kAccBufs, Cfg::kEpiWarp0, false>(p, sh, tmem, warp, lane, rank, abort);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (sh->fix_tile >= 0 && !sh->abort) {
    __threadfence();
    epilogue_fixup(p, sh->fix_tile, rank, sh->fix_nparts, sh->fix_mb, sh->fix_nb, threadIdx.x,
                   blockDim.x);
  }
}

// ------------------------------------------------------ CTA-pair kernel --
//
// Single-pass TF32 on the two SMs of a cluster acting as one tensor core
// (tcgen05 cta_group::2). The pair computes one unit tile, 256 n x 256 m of
// C^T, with one MMA stream issued by the even CTA: M = 256 (the MMA's A
// operand is B_tile^T, CTA r holding n rows 128 r .. 128 r + 127), N = 256
// (the MMA's B operand is the A tile, CTA r holding m rows 128 r ..) and
// K = 8. Each CTA's TMEM accumulates its own 128 n x 256 m, the same output
// tile tc_lsu_kernel gives one SM, so the schedule, epilogue and split-tile
// sums are shared with it.
//
// Both operands go from global memory to the tensor core by TMA alone: a
// K-major operand (A stored M x K, B stored N x K) as a box of BK k x 128
// rows with the 128-byte swizzle, an MN-major one (B stored K x N, A stored
// K x M) as four boxes of 32 mn x BK k with the 128-byte swizzle of 32-byte
// atoms, the layout kind::tf32 takes for MN-major operands. Each CTA's
// copies complete on the even CTA's stage barrier (which expects the bytes
// of both), the even CTA's commits release the stage in both, and nothing
// else crosses the pair per stage; the odd CTA's epilogue returns each
// accumulator to the even CTA once per tile.
template <int BK, int STAGES, bool OPA, bool OPB>
struct PairConfig {
  static_assert(BK == 32, "128-byte rows: one swizzle span per operand row");
  static constexpr int kHalfRows = 128;                          // rows of each operand per CTA
  static constexpr int kOpBytes = kHalfRows * BK * 4;            // one operand tile per CTA
  static constexpr int kAOffset = 0;                             // A rows (the MMA's B operand)
  static constexpr int kBtOffset = kOpBytes;                     // B^T rows (the MMA's A operand)
  static constexpr int kStageBytes = 2 * kOpBytes;
  static constexpr int kTileBytes = STAGES * kStageBytes;
  static constexpr int kAccBufs = 2;
  static constexpr int kMmaWarp = 1;
  static constexpr int kEpiWarp0 = 2;
  static constexpr int kThreads = 32 * (kEpiWarp0 + 4);
  // A operand (B^T) MN-major when B is stored K x N; B operand (A tile)
  // MN-major when A is stored K x M.
  static constexpr uint32_t kIdesc =
      idesc_tf32(2 * kTN, kTM) | (OPB ? 0u : 1u << 15) | (OPA ? 1u << 16 : 0u);
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kAccBufs * kTM <= static_cast<int>(kTmemCols), "TMEM budget");
};

// Shared-memory descriptor of k-step kk of an operand tile: K-major rows of
// 128 bytes (8-row swizzle atoms 1024 bytes apart, a k-step 32 bytes along
// the row), or MN-major chunks of 32 mn (BK * 128 bytes apart, 4-row groups
// 512 bytes apart, a k-step of 8 rows 1024 bytes on).
template <int BK, bool MN>
__device__ __forceinline__ uint64_t pair_operand_desc(uint32_t base, int kk) {
  if (MN) return smem_desc(base + kk * 1024, BK * 128, 512, 1);
  return smem_desc(base + kk * 32, 16, 1024, 2);
}

// Load this CTA's 128 rows x BK k of an operand whose rows start at `row0`
// (k from k0) into `dst`, completing on the even CTA's barrier `bar`. An
// MN-major operand is four chunks of 32 rows: one copy through a 3-D tensor
// map (`one_copy`), or one 2-D copy each. Fewer copies per stage run faster
// (timed: two copies per stage 0.90 of the peak at 4096^3, five 0.88, eight
// 0.72).
template <int BK, bool MN>
__device__ __forceinline__ void pair_load_operand(uint8_t *dst, const CUtensorMap *map,
                                                  uint32_t bar, int row0, int k0, bool one_copy) {
  if (MN && one_copy) {
    tma_load_3d_pair(dst, map, bar, 0, k0, row0 / 32);
  } else if (MN) {
#pragma unroll
    for (int c = 0; c < 4; ++c) tma_load_2d_pair(dst + c * BK * 128, map, bar, row0 + 32 * c, k0);
  } else {
    tma_load_2d_pair(dst, map, bar, k0, row0);
  }
}

//
// CS: a cluster holds p.ks pairs that share one unit tile (TcParams::ks);
// the pair of a CTA is its cluster rank with bit 0 cleared (pb), and its rank
// within the pair is bit 0.
// SCALED: built for alpha != 1 or beta != 0 (the whole-tile epilogue's
// scaled stores); the other instantiation stores the accumulators as they are.
template <int BK, int STAGES, bool OPA, bool OPB, bool CS = false, bool SCALED = false>
__global__ void __launch_bounds__(PairConfig<BK, STAGES, OPA, OPB>::kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const TcParams p) {
  using Cfg = PairConfig<BK, STAGES, OPA, OPB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcShared<STAGES> *sh = reinterpret_cast<TcShared<STAGES> *>(tiles + Cfg::kTileBytes);
  volatile int *abort = &sh->abort;

  const uint32_t warp = warp_index();
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t rank = CS ? (crank & 1u) : crank;  // rank within the pair
  const uint32_t pb = CS ? (crank & ~1u) : 0u;      // cluster rank of the pair's even CTA
  const uint16_t pair_mask = static_cast<uint16_t>(3u << pb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh->full[s], 1);   // even CTA: its producer's expect-tx; both CTAs' bytes
      mbar_init(&sh->empty[s], 1);  // the even CTA's commit, multicast to both
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->acc_full[a], 1);
      mbar_init(&sh->acc_empty[a], 8);  // even CTA: the four epilogue warps of each CTA
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    sh->fix_tile = -1;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc<2>(&sh->tmem_base, kTmemCols);
    tmem_relinquish<2>();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // barriers and TMEM of both CTAs set up before either signals the other
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  // Launched as a programmatic dependent: the set-up above overlapped the
  // previous grid (an operand copy, say); its results are needed from here on.
  grid_dependency_wait();

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_parity = 0;
      int issued = 0;
      bool ok = true;
      UnitIter it(p);
      WorkUnit u;
      while (ok && it.next(p, u)) {
        int mb, nb;
        tile_coords(p, u.tile, rank, mb, nb);
        const int m0 = mb * kTM + static_cast<int>(rank) * Cfg::kHalfRows;
        const int n0 = nb * kTN;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (issued++ == p.stall_kb) {  // self-test: stop feeding the pipeline
            ok = false;
            break;
          }
          if (!mbar_wait_bounded(&sh->empty[stage], phase ^ 1, p.timeout_ns, abort,
                                 &g_tc_status)) {
            ok = false;
            break;
          }
          uint8_t *st = tiles + stage * Cfg::kStageBytes;
          const uint32_t bar = mbar_cluster_addr(&sh->full[stage], pb);
          if (rank == 0) mbar_arrive_expect_tx(&sh->full[stage], 2 * Cfg::kStageBytes);
          pair_load_operand<BK, OPA>(st + Cfg::kAOffset, &tmap_a, bar, m0, kb * BK,
                                     p.a_one_copy != 0);
          pair_load_operand<BK, !OPB>(st + Cfg::kBtOffset, &tmap_b, bar, n0, kb * BK,
                                      p.b_one_copy != 0);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // On a timeout the even CTA lets the stages it armed land (both CTAs'
      // copies complete there) before the pair exits.
      if (!ok && rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) drain_wait(&sh->full[s], (armed_parity >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == Cfg::kMmaWarp) {
    // ------------------------------------------------- MMA (even CTA) --
    if (rank == 0 && lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      UnitIter it(p);
      WorkUnit u;
      while (ok && it.next(p, u)) {
        // Both CTAs' epilogues have drained this accumulator (the odd one's
        // arrivals come from the peer: acquire at cluster scope).
        if (!mbar_wait_bounded<true>(&sh->acc_empty[acc], acc_phase ^ 1, p.timeout_ns, abort,
                                     &g_tc_status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + kAccCol + acc * kTM;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&sh->full[stage], phase, p.timeout_ns, abort, &g_tc_status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t st = smem_addr(tiles + stage * Cfg::kStageBytes);
#pragma unroll
          for (int kk = 0; kk < BK / kUmmaK; ++kk)
            mma_tf32<2>(d_tmem, pair_operand_desc<BK, !OPB>(st + Cfg::kBtOffset, kk),
                        pair_operand_desc<BK, OPA>(st + Cfg::kAOffset, kk), Cfg::kIdesc,
                        (kb != u.kb0 || kk != 0) ? 1u : 0u);
          mma_commit_multicast<2>(&sh->empty[stage], pair_mask);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_multicast<2>(&sh->acc_full[acc], pair_mask);
        if (++acc == Cfg::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // Every MMA this thread issued completes before TMEM is released.
      mma_commit_multicast<2>(&sh->drain, static_cast<uint16_t>(1u << pb));
      drain_wait(&sh->drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    epilogue_role<Cfg::kAccBufs, Cfg::kEpiWarp0, true, CS, SCALED>(p, sh, tmem, warp, lane, rank, abort, pb,
                                                          reinterpret_cast<float *>(tiles));
  }

  // Neither CTA frees its TMEM or leaves while the pair's MMAs, copies or
  // arrivals may still reach it.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc<2>(tmem, kTmemCols);
  }
  if constexpr (CS) {
    // Every CTA's k-slice partial is in its slot (the cluster barrier above
    // orders the epilogue's stores before these reads).
    if (!sh->abort)
      cluster_split_sum<kClusterSumBatch>(p, reinterpret_cast<const float *>(tiles), crank,
                                          threadIdx.x, blockDim.x);
  }
  if (sh->fix_tile >= 0 && !sh->abort) {
    __threadfence();
    epilogue_fixup<16>(p, sh->fix_tile, rank, sh->fix_nparts, sh->fix_mb, sh->fix_nb, threadIdx.x,
                   blockDim.x);
  }
}

// -------------------------------------------------- CTA-pair 3xTF32 kernel --
//
// 3xTF32 on the two SMs of a cluster acting as one tensor core, for A stored
// M x K and B stored K x N or (OPB) N x K. The pair computes one unit tile, 256 n x 256 m
// of C^T, as in tc_pair_kernel: M = 256 (B_tile^T, CTA r holding n rows
// 128 r ..), N = 256 (the A tile, CTA r holding m rows 128 r ..), K = 8.
//
// Shared-memory traffic decides the design. With one SM per 128 n x 256 m
// output tile (an earlier TMA-fed design, 0.466 ms at 4096^3 against 0.398)
// every MMA reads 256 rows of its B operand and every SM splits a 256-row A
// tile, about 1.3 times the bytes per cycle shared memory can serve at full
// tensor rate; with the pair each SM reads and splits only its own 128 rows,
// for the same MMA work per SM.
//
// Per k-block of BK each CTA loads, by TMA on its own barriers, its 128 A
// rows x BK k (K-major, swizzled) into a ring of A stages and its B tile
// (BK k x 128 n row-major, or with OPB 128 n x BK k K-major and swizzled like
// A) into a ring of B slots. Its transform warps take
// the B tile into registers (freeing the slot), write B^T as hi and lo into
// a TMEM slot of its own (lane = n, one column per k) and split the A rows in
// place (hi) and into a sibling tile (lo). The even CTA's transform warps
// then arrive on its `ready` barrier; the odd CTA's arrive on a local barrier,
// and one relay thread passes the k-block on with a single remote arrive (a
// release at cluster scope, which orders the odd CTA's shared-memory and
// TMEM writes before the even CTA's MMAs). The even CTA issues B_lo*A_hi,
// B_hi*A_lo, B_hi*A_hi per k-step of 8 with A from TMEM and B from shared
// memory; its commits free the A stage and the TMEM slot in both CTAs.
//
// TMEM holds one 256-column accumulator and TST = 256 / (2 BK) B^T slots. The
// A ring is deeper than that, and B has a ring of its own, so the copies run
// ahead of the TMEM slots: a slot's round trip (the MMAs that read it, the
// transform of the next k-block, the hand-over) does not include a copy's
// latency.
// float4 loads per thread and part in flight in the 3xTF32 pair kernel's final
// split-tile sum (timed: 4 beats 16 by 1.5-2 us at 512^3-2048^3; the sum of a
// 128 KiB tile from parts just written by other SMs takes 5-10 us whatever
// the batch, bound by the latency of those loads).
constexpr int kPairExactFixBatch = 4;

template <int BK, int AST, int BST, int XW, bool OPB>
struct PairExactConfig {
  static_assert(BK == 16 || BK == 32, "BK");
  static constexpr int kHalfRows = 128;                          // A rows per CTA
  static constexpr int kRowBytes = BK * 4;                       // one K-major A row
  static constexpr int kAtomBytes = 8 * kRowBytes;               // 8-row swizzle atom (SBO)
  static constexpr uint32_t kLayout = BK == 32 ? 2u : 4u;        // 128- or 64-byte swizzle
  static constexpr int kABytes = kHalfRows * BK * 4;             // A rows (hi after the split)
  static constexpr int kALoOffset = kABytes;                     // A lo, same layout
  static constexpr int kAStageBytes = 2 * kABytes;
  // B tile: BK k x 128 n row-major (B stored K x N), or 128 n x BK k K-major
  // with A's swizzle (B stored N x K).
  static constexpr int kBBytes = BK * kTN * 4;
  static constexpr int kBRingOffset = AST * kAStageBytes;
  static constexpr int kTileBytes = AST * kAStageBytes + BST * kBBytes;
  static constexpr uint32_t kBtColsPerSlot = 2 * BK;             // B^T hi, then lo
  static constexpr int kTmemSlots = static_cast<int>((kTmemCols - kBtCol) / kBtColsPerSlot);
  static constexpr int kAccBufs = 1;
  static constexpr int kMmaWarp = 1;
  static constexpr int kEpiWarp0 = 2;
  static constexpr int kXformWarp0 = 6;
  static constexpr int kXformParts = XW / 4;                     // per TMEM lane quadrant
  static constexpr int kThreads = 32 * (kXformWarp0 + XW);
  static constexpr uint32_t kIdesc = idesc_tf32(2 * kTN, kTM);   // A from TMEM, B K-major
  static_assert(kAStageBytes % 1024 == 0 && kBRingOffset % 1024 == 0,
                "swizzled A stages keep 1024-byte alignment");
  static_assert(XW % 4 == 0 && BK % kXformParts == 0 && (BK / kXformParts) % 4 == 0,
                "transform partition");
  static_assert(AST >= kTmemSlots, "the A ring covers the TMEM slots");
};

// Shared state of the 3xTF32 pair kernel.
template <int AST, int BST, int TST>
struct alignas(8) PairExactShared {
  uint64_t full[AST];      // A stage loaded (TMA bytes)
  uint64_t empty[AST];     // A stage consumed by the MMAs (the even CTA's commit, both CTAs)
  uint64_t bfull[BST];     // B slot loaded (TMA bytes)
  uint64_t bempty[BST];    // B slot read by this CTA's transform warps
  uint64_t ready[TST];     // even CTA: k-block transformed in both CTAs
  uint64_t relay[TST];     // odd CTA: k-block transformed by its own transform warps
  uint64_t tfree[TST];     // TMEM slot's MMAs completed (the even CTA's commit, both CTAs)
  uint64_t acc_full[2];    // accumulator complete
  uint64_t acc_empty[2];   // accumulator drained by the epilogue warps of both CTAs
  uint64_t drain;          // every MMA of the pair has completed
  uint32_t tmem_base;
  int abort;
  int sk_last;
  int fix_tile, fix_nparts, fix_mb, fix_nb;
};

// Ring position: index and phase parity of a ring of N entries.
template <int N>
struct RingPos {
  uint32_t idx = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++idx == N) {
      idx = 0;
      phase ^= 1;
    }
  }
};

// CS: as for tc_pair_kernel, p.ks pairs per cluster share one unit tile.
// SCALED: as for tc_pair_kernel.
template <int BK, int AST, int BST, int XW, bool OPB, bool CS = false, bool SCALED = false>
__global__ void __launch_bounds__(PairExactConfig<BK, AST, BST, XW, OPB>::kThreads, 1)
    tc_pair_exact_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b, const TcParams p) {
  using Cfg = PairExactConfig<BK, AST, BST, XW, OPB>;
  constexpr int TST = Cfg::kTmemSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto *sh = reinterpret_cast<PairExactShared<AST, BST, TST> *>(tiles + Cfg::kTileBytes);
  volatile int *abort = &sh->abort;

  const uint32_t warp = warp_index();
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t rank = CS ? (crank & 1u) : crank;  // rank within the pair
  const uint32_t pb = CS ? (crank & ~1u) : 0u;      // cluster rank of the pair's even CTA
  const uint16_t pair_mask = static_cast<uint16_t>(3u << pb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < AST; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int b = 0; b < BST; ++b) {
      mbar_init(&sh->bfull[b], 1);
      mbar_init(&sh->bempty[b], XW);
    }
    for (int t = 0; t < TST; ++t) {
      mbar_init(&sh->ready[t], XW + 1);  // the even CTA's transform warps, the odd CTA's relay
      mbar_init(&sh->relay[t], XW);
      mbar_init(&sh->tfree[t], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->acc_full[a], 1);
      mbar_init(&sh->acc_empty[a], 8);   // even CTA: the four epilogue warps of each CTA
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    sh->fix_tile = -1;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmap_a);
    tma_prefetch_map(&tmap_b);
  }
  if (warp == Cfg::kMmaWarp) {
    tmem_alloc<2>(&sh->tmem_base, kTmemCols);
    tmem_relinquish<2>();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // barriers and TMEM of both CTAs set up before either signals the other
  tc_fence_after_sync();
  const uint32_t tmem = sh->tmem_base;
  // Launched as a programmatic dependent: the set-up above overlapped the
  // previous grid (an operand copy, say); its results are needed from here on.
  grid_dependency_wait();

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      RingPos<AST> a;
      RingPos<BST> b;
      uint32_t armed = 0, armed_parity = 0, barmed = 0, barmed_parity = 0;
      int issued = 0;
      bool ok = true;
      StreamGate gate;
      UnitIter it(p);
      WorkUnit u;
      while (ok && it.next(p, u)) {
        int mb, nb;
        tile_coords(p, u.tile, rank, mb, nb);
        const int m0 = mb * kTM + static_cast<int>(rank) * Cfg::kHalfRows;
        const int n0 = nb * kTN;
        if (!gate.tile(p, mb, abort)) {
          ok = false;
          break;
        }
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (issued++ == p.stall_kb) {  // self-test: stop feeding the pipeline
            ok = false;
            break;
          }
          if (!gate.kblock(p, kb, abort)) {
            ok = false;
            break;
          }
          if (!mbar_wait_bounded(&sh->empty[a.idx], a.phase ^ 1, p.timeout_ns, abort,
                                 &g_tc_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh->full[a.idx], Cfg::kABytes);
          tma_load_2d(tiles + a.idx * Cfg::kAStageBytes, &tmap_a, &sh->full[a.idx], kb * BK, m0);
          armed |= 1u << a.idx;
          armed_parity = (armed_parity & ~(1u << a.idx)) | (a.phase << a.idx);
          a.next();
          if (!mbar_wait_bounded(&sh->bempty[b.idx], b.phase ^ 1, p.timeout_ns, abort,
                                 &g_tc_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh->bfull[b.idx], Cfg::kBBytes);
          if (OPB)
            tma_load_2d(tiles + Cfg::kBRingOffset + b.idx * Cfg::kBBytes, &tmap_b,
                        &sh->bfull[b.idx], kb * BK, n0);
          else
            tma_load_2d(tiles + Cfg::kBRingOffset + b.idx * Cfg::kBBytes, &tmap_b,
                        &sh->bfull[b.idx], n0, kb * BK);
          barmed |= 1u << b.idx;
          barmed_parity = (barmed_parity & ~(1u << b.idx)) | (b.phase << b.idx);
          b.next();
        }
      }
      // Let every copy this thread issued land before the CTA exits.
      if (!ok) {
        for (int s = 0; s < AST; ++s)
          if (armed & (1u << s)) drain_wait(&sh->full[s], (armed_parity >> s) & 1u, p.timeout_ns);
        for (int s = 0; s < BST; ++s)
          if (barmed & (1u << s))
            drain_wait(&sh->bfull[s], (barmed_parity >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == Cfg::kMmaWarp) {
    if (rank == 0 && lane == 0) {
      // ----------------------------------------------- MMA (even CTA) --
      RingPos<AST> a;
      RingPos<TST> t;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      UnitIter it(p);
      WorkUnit u;
      while (ok && it.next(p, u)) {
        // Both CTAs' epilogues have drained the accumulator.
        if (!mbar_wait_bounded<true>(&sh->acc_empty[acc], acc_phase ^ 1, p.timeout_ns, abort,
                                     &g_tc_status)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + kAccCol + acc * kTM;
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          // Both CTAs' transform warps are done with the k-block (the odd
          // CTA's relay arrives from the peer: acquire at cluster scope).
          if (!mbar_wait_bounded<true>(&sh->ready[t.idx], t.phase, p.timeout_ns, abort,
                                       &g_tc_status)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_hi = smem_addr(tiles + a.idx * Cfg::kAStageBytes);
          const uint32_t bt_hi = tmem + kBtCol + t.idx * Cfg::kBtColsPerSlot;
#pragma unroll
          for (int kk = 0; kk < BK / kUmmaK; ++kk) {
            const uint64_t da = smem_desc(a_hi + kk * 32, 16, Cfg::kAtomBytes, Cfg::kLayout);
            const uint64_t da_lo =
                smem_desc(a_hi + Cfg::kALoOffset + kk * 32, 16, Cfg::kAtomBytes, Cfg::kLayout);
            const uint32_t accumulate = (kb != u.kb0 || kk != 0) ? 1u : 0u;
            mma_tf32_ts<2>(d_tmem, bt_hi + BK + kk * kUmmaK, da, Cfg::kIdesc, accumulate);
            mma_tf32_ts<2>(d_tmem, bt_hi + kk * kUmmaK, da_lo, Cfg::kIdesc, 1);
            mma_tf32_ts<2>(d_tmem, bt_hi + kk * kUmmaK, da, Cfg::kIdesc, 1);
          }
          mma_commit_multicast<2>(&sh->empty[a.idx], pair_mask);
          mma_commit_multicast<2>(&sh->tfree[t.idx], pair_mask);
          a.next();
          t.next();
        }
        if (!ok) break;
        mma_commit_multicast<2>(&sh->acc_full[acc], pair_mask);
        if (++acc == Cfg::kAccBufs) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // Every MMA this thread issued completes before TMEM is released.
      mma_commit_multicast<2>(&sh->drain, static_cast<uint16_t>(1u << pb));
      drain_wait(&sh->drain, 0, p.timeout_ns);
    } else if (rank == 1 && lane == 0) {
      // ---------------------------------------------- relay (odd CTA) --
      // Once all of this CTA's transform warps are done with a k-block, one
      // release at cluster scope passes it on to the even CTA's MMAs (eight
      // warps each arriving remotely took twice as long per k-block).
      RingPos<TST> t;
      bool ok = true;
      UnitIter it(p);
      WorkUnit u;
      while (ok && it.next(p, u)) {
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait_bounded(&sh->relay[t.idx], t.phase, p.timeout_ns, abort, &g_tc_status)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(&sh->ready[t.idx], pb);
          t.next();
        }
      }
    }
    __syncwarp();
  } else if (warp < Cfg::kEpiWarp0 + 4) {
    // --------------------------------------------------------- epilogue --
    epilogue_role<Cfg::kAccBufs, Cfg::kEpiWarp0, true, CS, SCALED>(p, sh, tmem, warp, lane, rank, abort, pb,
                                                          reinterpret_cast<float *>(tiles));
  } else {
    // --------------------------------------------------------- transform --
    // Warp (quad, part) moves k in [part * W, (part + 1) * W), W = BK / parts,
    // of B^T rows n = 32 quad + lane into TMEM as hi and lo; all of them
    // split this CTA's A rows.
    const uint32_t quad = warp & 3;
    const uint32_t part = (warp - Cfg::kXformWarp0) >> 2;
    const int xt = threadIdx.x - Cfg::kXformWarp0 * 32;
    constexpr int kW = BK / Cfg::kXformParts;
    RingPos<AST> a;
    RingPos<BST> b;
    RingPos<TST> t;
    bool ok = true;
    UnitIter it(p);
    WorkUnit u;
    while (ok && it.next(p, u)) {
      for (int kb = u.kb0; kb < u.kb1; ++kb) {
        // B tile into registers; the slot can then be refilled.
        if (!warp_wait(&sh->bfull[b.idx], b.phase, p, abort)) {
          ok = false;
          break;
        }
        const uint8_t *bslot = tiles + Cfg::kBRingOffset + b.idx * Cfg::kBBytes;
        float v[kW];
        if constexpr (OPB) {
          // Row n = 32 quad + lane of the K-major tile; this part's kW k as
          // 16-byte chunks of the swizzled row.
          const int n = quad * 32 + lane;
#pragma unroll
          for (int c = 0; c < kW / 4; ++c) {
            const float4 x = *reinterpret_cast<const float4 *>(
                bslot + swizzle_a<BK>(n * Cfg::kRowBytes + (part * kW + c * 4) * 4));
            v[c * 4 + 0] = x.x;
            v[c * 4 + 1] = x.y;
            v[c * 4 + 2] = x.z;
            v[c * 4 + 3] = x.w;
          }
        } else {
          // Column n = 32 quad + lane of the row-major tile.
          const float *bs =
              reinterpret_cast<const float *>(bslot) + part * kW * kTN + quad * 32 + lane;
#pragma unroll
          for (int k = 0; k < kW; ++k) v[k] = bs[k * kTN];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->bempty[b.idx]);
        b.next();
        // B^T into the TMEM slot once the MMAs that last read it are done.
        if (!warp_wait(&sh->tfree[t.idx], t.phase ^ 1, p, abort)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t col =
            tmem + ((quad * 32) << 16) + kBtCol + t.idx * Cfg::kBtColsPerSlot + part * kW;
        bt_to_tmem<kW, true>(col, col + BK, v);
        // Split the A rows: hi in place, lo in the sibling tile.
        if (!warp_wait(&sh->full[a.idx], a.phase, p, abort)) {
          ok = false;
          break;
        }
        float4 *raw = reinterpret_cast<float4 *>(tiles + a.idx * Cfg::kAStageBytes);
        float4 *lo =
            reinterpret_cast<float4 *>(tiles + a.idx * Cfg::kAStageBytes + Cfg::kALoOffset);
#pragma unroll
        for (int i = xt; i < Cfg::kABytes / 16; i += 32 * XW) {
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
        // The MMAs read the split tile through the async proxy and B^T from
        // TMEM; both are ordered before the arrival.
        fence_proxy_async_smem();
        tmem_store_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(rank == 0 ? &sh->ready[t.idx] : &sh->relay[t.idx]);
        a.next();
        t.next();
      }
    }
  }

  // Neither CTA frees its TMEM or leaves while the pair's MMAs, copies or
  // arrivals may still reach it.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == Cfg::kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc<2>(tmem, kTmemCols);
  }
  stream_release(p, sh->abort != 0);
  if constexpr (CS) {
    // Every CTA's k-slice partial is in its slot (the cluster barrier above
    // orders the epilogue's stores before these reads).
    if (!sh->abort)
      cluster_split_sum<kClusterSumBatch>(p, reinterpret_cast<const float *>(tiles), crank,
                                          threadIdx.x, blockDim.x);
  }
  if (sh->fix_tile >= 0 && !sh->abort) {
    __threadfence();
    epilogue_fixup<kPairExactFixBatch>(p, sh->fix_tile, rank, sh->fix_nparts, sh->fix_mb,
                                       sh->fix_nb, threadIdx.x, blockDim.x);
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
  uint32_t b0, b1, swizzle, rank;
  bool operator==(const MapKey &o) const {
    return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && pitch == o.pitch && b0 == o.b0 &&
           b1 == o.b1 && swizzle == o.swizzle && rank == o.rank;
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

// Encode (or find in a small cache) an fp32 tensor map with zero fill outside
// the matrix. rank 2: a row-major matrix (d0 = columns, d1 = rows, row pitch
// `pitch` bytes), b0 x b1 box. rank 3: the same matrix seen as chunks of 32
// columns -- dims {32, d1, d0 / 32}, strides {pitch, 128 bytes}, box {32, b1,
// b0 / 32} -- so that one copy brings b0 columns as b0 / 32 chunks of 32 x
// b1, one after another (d0 must be a multiple of 32: every chunk is then
// inside the rows).
bool get_map_rank(const void *ptr, uint64_t d0, uint64_t d1, uint64_t pitch_bytes, uint32_t b0,
                  uint32_t b1, CUtensorMapSwizzle swizzle, uint32_t rank, CUtensorMap *out) {
  static MapCache cache;
  const MapKey key{ptr, d0, d1, pitch_bytes, b0, b1, static_cast<uint32_t>(swizzle), rank};
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
  cuuint64_t dims[3] = {d0, d1, 1};
  cuuint64_t strides[2] = {pitch_bytes, 0};
  cuuint32_t box[3] = {b0, b1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (rank == 3) {
    if (d0 % 32 != 0 || b0 % 32 != 0) return false;
    dims[0] = 32;
    dims[2] = d0 / 32;
    strides[1] = 128;
    box[0] = 32;
    box[2] = b0 / 32;
  }
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void *>(ptr), dims, strides, box,
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

// 2-D fp32 tensor map over a row-major matrix (d0 = columns, d1 = rows) with a
// b0 x b1 box, the given swizzle, and zero fill outside the matrix.
bool get_map(const void *ptr, uint64_t d0, uint64_t d1, uint64_t pitch_bytes, uint32_t b0,
             uint32_t b1, CUtensorMapSwizzle swizzle, CUtensorMap *out) {
  return get_map_rank(ptr, d0, d1, pitch_bytes, b0, b1, swizzle, 2, out);
}

// Smallest stream-K chunk, in k: shorter chunks spend more time filling the
// pipeline and more bytes on partial tiles than they save. One TF32 pass
// does a third of the MMA work per k of 3xTF32, so splitting pays only for
// longer chunks (timed on 512 x 512 x 8192, 1024^3, 1024 x 1024 x 8192,
// 2048^3, 2048 x 2048 x 8192, 1000 x 1531 x 777 and 3072^3: 2048 k before a
// split is worth it in tf32 -- at 1024 k 2048^3 takes 49 us instead of 31 --
// and 256 k in exact mode).
constexpr int kMinChunkKExact = 256;
constexpr int kMinChunkKTf32 = 2048;
// What splitting the last wave's tiles costs the 3xTF32 pair kernel, in k of
// MMA work: writing the partial tiles and the final sums (timed with 0, 448,
// 768 and 1024: at 768, 2048^3 runs its 64 tiles whole on 64 pairs, 74 -> 67
// us, 1000 x 1531 x 777 46 -> 44 us, 512^3 28.5 -> 27 us; 4096^3 and 8192 x
// 11008 x 4096 keep their split last wave; 1024 made 1024^3 slower).
constexpr int kSplitCostKExact = 768;
// Most CTAs sharing one split tile: the last of them sums every part alone.
constexpr int kMaxSplit = 8;

struct Schedule {
  int grid, dp_tiles, sk_share, sk_ctas;
  bool splits;  // some tile's k range is shared by two or more chunks
};

// Data-parallel waves plus a stream-K tail, over G workers (SMs, or CTA
// pairs). With T tiles of KB k-blocks and T mod G != 0:
//  - balanced (full_waves = false): all but the last full wave are dealt
//    whole; the k-blocks of the remaining G + T mod G tiles are cut into
//    equal contiguous chunks over the G workers. Each chunk is then at least
//    one tile long, so a split tile has at most two parts, and every worker
//    ends up with about T * KB / G k-blocks.
//  - full_waves: every full wave is dealt whole and only the T mod G tiles of
//    the last one are split, over as many workers as chunks of at least
//    min_chunk k-blocks allow. The tail runs on fewer workers, which is faster
//    for a kernel bound by the operand traffic out of L2 (each worker left
//    running gets a larger share of it) but not for one bound by its MMAs.
// With fewer tiles than workers everything is stream-K, with chunks of at
// least min_chunk k-blocks and at most kMaxSplit parts per tile.
Schedule make_schedule(int tiles, int kb, int sms, int min_chunk, bool full_waves,
                       int split_cost = 0) {
  Schedule s;
  min_chunk = min_chunk < 1 ? 1 : min_chunk;
  s.dp_tiles = (tiles >= sms && tiles % sms != 0) ? (tiles / sms - (full_waves ? 0 : 1)) * sms
               : (tiles >= sms ? tiles : 0);
  // Full waves: the last R = tiles - dp_tiles tiles are dealt whole as well
  // when splitting them would save less than it costs: (1 - R / G) of a
  // tile's kb k-blocks against split_cost k-blocks for writing and summing
  // partial tiles.
  if (full_waves && tiles > s.dp_tiles &&
      static_cast<long long>(kb) * (sms - (tiles - s.dp_tiles)) <
          static_cast<long long>(split_cost) * sms)
    s.dp_tiles = tiles;
  const int split = tiles - s.dp_tiles;
  if (split == 0) {
    s.grid = sms < tiles ? sms : tiles;
    s.sk_share = 1;
    s.sk_ctas = 0;
    s.splits = false;
    return s;
  }
  const long long total = static_cast<long long>(split) * kb;
  long long ctas;
  if (split >= sms) {
    ctas = sms;  // one chunk per SM, each at least a tile long
  } else {
    ctas = total / min_chunk;
    if (ctas > sms) ctas = sms;
    // A tile meets at most floor((kb - 1) / share) + 2 chunks; a share of at
    // least ceil(kb / (kMaxSplit - 1)) keeps that at kMaxSplit.
    const long long min_share = (kb + kMaxSplit - 2) / (kMaxSplit - 1);
    if (ctas > total / min_share) ctas = total / min_share;
    if (ctas < split) ctas = split;  // at least one CTA per tile
    if (ctas > total) ctas = total;
  }
  s.sk_share = static_cast<int>((total + ctas - 1) / ctas);
  s.sk_ctas = static_cast<int>((total + s.sk_share - 1) / s.sk_share);
  // Chunks that are whole multiples of a tile never split one.
  s.splits = s.sk_share % kb != 0;
  s.grid = (split >= sms || s.dp_tiles > 0) ? sms : s.sk_ctas;
  return s;
}

// Whether the pair kernels take their stream-K chunk before their whole
// tiles (TcParams::sk_first). The split-tile sums then run in the epilogue
// while the MMAs go on with whole tiles, instead of after the last tile. The
// 3xTF32 kernel gains at every size (4096^3: 394.7 -> 385.8 us,
// 3328 x 1536 x 4096: 158 -> 144 us, 8192 x 11008 x 4096: -0.6 %). For one
// TF32 pass, whose copies compete with the sums for L2 bandwidth, it pays
// only while the tail is a large part of the work (4096^3, three whole
// waves: 162.5 -> 159.3 us; 3328 x 1536 x 4096, one: 78.5 -> 70.8 us;
// 8192 x 11008 x 4096, 18: 776 -> 785 us): at most 8 whole waves.
bool split_chunk_first(const Schedule &sch, int workers, bool exact, bool pair) {
  if (!pair) return false;
  return exact || sch.dp_tiles <= 8 * workers;
}

// Tile counts of a launch: unit tiles of kTM rows x CL * kTN columns, k-blocks
// of BK.
void set_tiles(TcParams &p, int64_t M, int64_t N, int64_t K, int bk, int cl) {
  p.num_m_blocks = static_cast<int>((M + kTM - 1) / kTM);
  p.num_n_blocks = static_cast<int>((N + kTN - 1) / kTN);
  p.num_k_blocks = static_cast<int>((K + bk - 1) / bk);
  p.cl = cl;
  p.num_nu_blocks = (p.num_n_blocks + cl - 1) / cl;
  p.num_tiles = p.num_m_blocks * p.num_nu_blocks;
}

// The schedule policy of each kernel (see make_schedule and the constants
// above), on `workers` clusters.
Schedule schedule_for(const TcParams &p, int workers, int bk, bool exact, bool pair) {
  // Full waves for the pair kernels, balanced for tc_lsu_kernel (timed at
  // 4096^3, 5120^3, 2560 x 2560 x 4096 and 8192 x 11008 x 4096: +5-6 % for
  // the TF32 pair kernel, which is bound by operand traffic from L2, +3 % at
  // 4096^3 for the 3xTF32 pair kernel, whose split tiles then have fewer
  // parts to sum, and -3 % for an earlier one-SM 3xTF32 kernel).
  return make_schedule(p.num_tiles, p.num_k_blocks, workers,
                       (exact ? kMinChunkKExact : kMinChunkKTf32) / bk, pair,
                       pair && exact ? kSplitCostKExact / bk : 0);
}

// The kernel a launch plan runs: tc_lsu_kernel, or with PAIR a CTA-pair
// kernel.
template <int BK, int STAGES, bool EXACT, bool LSU, int CL, bool OPB, bool OPA, int BST, bool PAIR,
          bool CS = false, bool SCALED = false>
struct KernelOf {
  static_assert(LSU && CL == 1 && BST == 0 && !CS,
                "tc_lsu_kernel: plain-load producers, one SM per tile");
  using Cfg = TcConfig<BK, STAGES, EXACT, OPB>;
  static constexpr int kThreads = Cfg::kThreads;
  static constexpr int kSmemBytes =
      Cfg::kTileBytes + static_cast<int>(sizeof(TcShared<STAGES>)) + 1024;
  static constexpr auto kernel = tc_lsu_kernel<BK, STAGES, EXACT, OPB, OPA>;
};

template <int BK, int STAGES, bool OPA, bool OPB, bool CS, bool SCALED>
struct PairTf32Kernel {
  using Cfg = PairConfig<BK, STAGES, OPA, OPB>;
  static_assert(Cfg::kTileBytes >= kTM * kTN * 4, "a cluster-split band fits the stages");
  static constexpr int kThreads = Cfg::kThreads;
  static constexpr int kSmemBytes =
      Cfg::kTileBytes + static_cast<int>(sizeof(TcShared<STAGES>)) + 1024;
  static constexpr auto kernel = tc_pair_kernel<BK, STAGES, OPA, OPB, CS, SCALED>;
};

// Transform warps per CTA of the 3xTF32 pair kernel (16 time the same).
constexpr int kPairExactXform = 8;

template <int BK, int AST, int BST, int XW, bool OPB, bool CS, bool SCALED>
struct PairExactKernel {
  using Cfg = PairExactConfig<BK, AST, BST, XW, OPB>;
  static_assert(Cfg::kBRingOffset >= kTM * kTN * 4, "a cluster-split band fits the A ring");
  static constexpr int kThreads = Cfg::kThreads;
  static constexpr int kSmemBytes =
      Cfg::kTileBytes +
      static_cast<int>(sizeof(PairExactShared<AST, BST, Cfg::kTmemSlots>)) + 1024;
  static constexpr auto kernel = tc_pair_exact_kernel<BK, AST, BST, XW, OPB, CS, SCALED>;
};

// PAIR: the CTA-pair kernels, one TF32 pass (every layout) or 3xTF32 (A
// stored M x K, B in either storage).
// With EXACT, STAGES counts A stages and BST the B slots.
// CS: the cluster-split variant (TcParams::ks pairs per cluster and tile).
template <int BK, int STAGES, bool EXACT, bool LSU, int CL, bool OPB, bool OPA, int BST, bool CS,
          bool SCALED>
struct KernelOf<BK, STAGES, EXACT, LSU, CL, OPB, OPA, BST, true, CS, SCALED>
    : std::conditional_t<EXACT, PairExactKernel<BK, STAGES, BST, kPairExactXform, OPB, CS, SCALED>,
                         PairTf32Kernel<BK, STAGES, OPA, OPB, CS, SCALED>> {
  static_assert(!LSU && CL == 2 && (EXACT ? BST > 0 : BST == 0), "the pair kernels are fed by TMA");
  static_assert(!EXACT || !OPA, "3xTF32 pairs: A stored M x K");
};

// Cluster split (TcParams::ks): worth it only when the k range each pair no
// longer computes, kb (1 - 1 / ks), outweighs the exchange of partial tiles
// (moving the accumulator out of TMEM, a cluster barrier, reading 64-96 KiB
// of the other pairs' partials through L2 at about 56 GB/s per SM): at least
// 128 k of 3xTF32 work or 768 k of one TF32 pass (timed: with 128 k instead
// of 256, 512 x 512 x 256 20.1 -> 17.5 us, 1024 x 1024 x 256 20.5 -> 17.9 us,
// 300 x 700 x 300 22.6 -> 18.1 us; one TF32 pass with 384 k instead of 768,
// 512^3 15.0 -> 16.2 us, 1000 x 1532 x 776 19.4 -> 19.8 us).
constexpr int kClusterSplitSavedKExact = 128;
constexpr int kClusterSplitSavedKTf32 = 768;

// Pairs per unit tile for a problem of `tiles` unit tiles of kb k-blocks on
// `pairs` CTA pairs: as many as there are pairs per tile, up to
// kClusterSplitMax, if that saves enough k per pair; < 2 means no cluster
// split (the stream-K schedule applies). Host and device code.
__host__ __device__ inline int cluster_split_ks(int tiles, int kb, int pairs, int bk, bool exact) {
  int ks = pairs / (tiles > 0 ? tiles : 1);
  if (ks > kClusterSplitMax) ks = kClusterSplitMax;
  if (ks > kb) ks = kb;
  if (ks < 2) return 1;
  const long long saved_k = static_cast<long long>(kb) * bk * (ks - 1) / ks;
  return saved_k >= (exact ? kClusterSplitSavedKExact : kClusterSplitSavedKTf32) ? ks : 1;
}

// Everything a launch needs except the stream-K workspace. CS: the
// cluster-split launch of a pair kernel; prepare() sets p.ks = 1 when the
// problem does not take it, and the caller then launches the plain plan.
template <int BK, int STAGES, bool EXACT, bool LSU, int CL, bool OPB, bool OPA = false,
          int BST = 0, bool PAIR = false, bool CS = false, bool SCALED = false>
struct LaunchPlan {
  static_assert(!CS || PAIR, "cluster split: pair kernels only");
  using K = KernelOf<BK, STAGES, EXACT, LSU, CL, OPB, OPA, BST, PAIR, CS, SCALED>;
  TcParams p;
  Schedule sch;
  CUtensorMap map_a, map_b;
  int smem_bytes = 0;
  size_t counter_bytes = 0, partial_bytes = 0;  // workspace, 0 if no tile is split
  // Set before prepare() for a streamed launch (pair kernels, CS = false).
  const StreamFeed *feed = nullptr;

  int prepare(const GemmArgs &a, int sm_count) {
    auto kernel = K::kernel;
    smem_bytes = K::kSmemBytes;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kErrLaunch;
    static bool attr_set[64] = {};
    static std::mutex attr_mu;
    {
      std::lock_guard<std::mutex> g(attr_mu);
      if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess)
          return kErrLaunch;
        attr_set[dev] = true;
      }
    }
    std::memset(&map_a, 0, sizeof(map_a));
    std::memset(&map_b, 0, sizeof(map_b));
    p.a_one_copy = 0;
    p.b_one_copy = 0;
    if constexpr (PAIR && !EXACT) {
      // K-major operands: BK k x 128 rows, 128-byte swizzle. MN-major ones
      // (A stored K x M, B stored K x N): 32 mn x BK k, 32-byte atoms.
      const CUtensorMapSwizzle k_sw = CU_TENSOR_MAP_SWIZZLE_128B;
      const CUtensorMapSwizzle mn_sw = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
      p.a_one_copy = OPA && a.M % 32 == 0;
      p.b_one_copy = !OPB && a.N % 32 == 0;
      if (!(OPA ? get_map_rank(a.A, a.M, a.K, a.lda * 4, p.a_one_copy ? 128 : 32, BK, mn_sw,
                               p.a_one_copy ? 3 : 2, &map_a)
                : get_map(a.A, a.K, a.M, a.lda * 4, BK, 128, k_sw, &map_a)))
        return kErrLaunch;
      if (!(OPB ? get_map(a.B, a.K, a.N, a.ldb * 4, BK, 128, k_sw, &map_b)
                : get_map_rank(a.B, a.N, a.K, a.ldb * 4, p.b_one_copy ? 128 : 32, BK, mn_sw,
                               p.b_one_copy ? 3 : 2, &map_b)))
        return kErrLaunch;
    } else if constexpr (!LSU) {
      const CUtensorMapSwizzle sw_a =
          BK == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
      // Each CTA of the 3xTF32 pair loads its own half of the A tile.
      if (!get_map(a.A, a.K, a.M, a.lda * 4, BK, kTM / CL, sw_a, &map_a)) return kErrLaunch;
      if (OPB) {
        // B stored N x K: a K-major BK x 128 box with A's swizzle.
        if (!get_map(a.B, a.K, a.N, a.ldb * 4, BK, kTN, sw_a, &map_b)) return kErrLaunch;
      } else if (!get_map(a.B, a.N, a.K, a.ldb * 4, kTN, BK, CU_TENSOR_MAP_SWIZZLE_NONE, &map_b)) {
        return kErrLaunch;
      }
    }
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
    p.partial_extent = 0;
    p.counter_extent = 0;
    set_tiles(p, a.M, a.N, a.K, BK, CL);
    // Generous: a stage takes microseconds; one tile's mainloop about K * 25 ns.
    p.timeout_ns = 2000000000ull + static_cast<unsigned long long>(a.K) * 2000ull;
    p.stall_kb = -1;
    p.ks = 1;
    p.sk_first = 0;
    p.sk_partials = nullptr;
    p.sk_counters = nullptr;
    p.group_m = kGroupM;
    p.stream_a_ready = nullptr;
    p.stream_b_ready = nullptr;
    p.stream_c_done = nullptr;
    p.stream_epoch = 0;
    p.stream_kb_split = 0;
    p.stream_group = 1;
    if constexpr (CS) {
      // ks pairs per unit tile, if the problem has few enough tiles and all
      // its clusters of 2 ks CTAs can be resident at once (checked once per
      // device and ks).
      int ks = cluster_split_ks(p.num_tiles, p.num_k_blocks, sm_count / 2, BK, EXACT);
      static int fits[64][kClusterSplitMax + 1] = {};
      static std::mutex fits_mu;
      for (; ks >= 2; --ks) {
        std::lock_guard<std::mutex> g(fits_mu);
        if (fits[dev][ks] == 0) {
          cudaLaunchConfig_t qc = {};
          qc.gridDim = dim3(2 * ks, 1, 1);
          qc.blockDim = dim3(K::kThreads, 1, 1);
          qc.dynamicSmemBytes = smem_bytes;
          cudaLaunchAttribute attr[1];
          attr[0].id = cudaLaunchAttributeClusterDimension;
          attr[0].val.clusterDim.x = 2 * ks;
          attr[0].val.clusterDim.y = 1;
          attr[0].val.clusterDim.z = 1;
          qc.attrs = attr;
          qc.numAttrs = 1;
          int clusters = 0;
          if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &qc) != cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
          }
          fits[dev][ks] = clusters > 0 ? clusters : -1;
        }
        if (fits[dev][ks] >= p.num_tiles) break;
      }
      if (ks < 2) return kOk;  // p.ks == 1: not taken
      p.ks = ks;
      sch.grid = p.num_tiles * ks;  // pairs
      sch.dp_tiles = 0;
      sch.sk_share = 1;
      sch.sk_ctas = 0;
      sch.splits = false;
      p.dp_tiles = 0;
      p.sk_share = 1;
      p.sk_ctas = 0;
      // One kTM x kTN partial slot per CTA, no counters.
      partial_bytes = static_cast<size_t>(sch.grid) * CL * kTM * kTN * 4;
      return kOk;
    }
    // Workers: clusters that can be resident at once (the placement of CTA
    // pairs may leave some SMs unpaired).
    static int workers_cached[64] = {};
    static std::mutex workers_mu;
    int workers = sm_count / CL;
    if (CL > 1) {
      std::lock_guard<std::mutex> g(workers_mu);
      if (workers_cached[dev] == 0) {
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(CL * workers, 1, 1);
        qc.blockDim = dim3(K::kThreads, 1, 1);
        qc.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        qc.attrs = attr;
        qc.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &qc) != cudaSuccess || clusters <= 0)
          return kErrLaunch;
        workers_cached[dev] = clusters < workers ? clusters : workers;
      }
      workers = workers_cached[dev];
    }
    if (feed != nullptr) {
      // Streamed launch: whole unit tiles dealt round-robin in row-major
      // order (the order A arrives in), no tile split, no workspace.
      if (!PAIR || !EXACT || CS) return kErrInvalidArg;
      p.group_m = 1;
      p.stream_a_ready = feed->a_ready;
      p.stream_b_ready = feed->b_ready;
      p.stream_c_done = feed->c_done;
      p.stream_epoch = feed->epoch;
      p.stream_kb_split = feed->kb_split;
      p.stream_group = feed->group;
      if (p.stream_group < 1) return kErrInvalidArg;
      if (feed->timeout_ns > 0) p.timeout_ns = feed->timeout_ns;
      sch.grid = workers < p.num_tiles ? workers : p.num_tiles;
      sch.dp_tiles = p.num_tiles;
      sch.sk_share = 1;
      sch.sk_ctas = 0;
      sch.splits = false;
      p.dp_tiles = p.num_tiles;
      p.sk_share = 1;
      p.sk_ctas = 0;
      return kOk;
    }
    sch = schedule_for(p, workers, BK, EXACT, PAIR);
    p.dp_tiles = sch.dp_tiles;
    p.sk_share = sch.sk_share;
    p.sk_ctas = sch.sk_ctas;
    p.sk_first = split_chunk_first(sch, workers, EXACT, PAIR) ? 1 : 0;
    const int split_tiles = p.num_tiles - p.dp_tiles;
    if (split_tiles > 0 && sch.splits) {
      counter_bytes = (static_cast<size_t>(split_tiles) * CL * 4 + 255) / 256 * 256;
      partial_bytes = static_cast<size_t>(sch.sk_ctas) * 2 * CL * kTM * kTN * 4;
    }
    return kOk;
  }

  size_t workspace_bytes() const { return counter_bytes + partial_bytes; }

  // Point the schedule at a workspace of counter_bytes + partial_bytes.
  void set_workspace(void *ws) {
    p.sk_counters = static_cast<unsigned *>(ws);
    p.sk_partials = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + counter_bytes);
    p.counter_extent = static_cast<long long>(counter_bytes / 4);
    p.partial_extent = static_cast<long long>(partial_bytes / 4);
  }

  int launch(cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sch.grid * CL, 1, 1);
    cfg.blockDim = dim3(K::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    // A programmatic dependent of the previous grid on the stream: the launch
    // and set-up overlap its tail (the kernels wait for it before they touch
    // memory). After the operand copies of 1000 x 1531 x 777 (pitches of 777
    // and 1531 floats): 37.3 -> 34.7 us exact, 29.4 -> 26.7 us tf32.
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CS ? CL * p.ks : CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL > 1 ? 2 : 1;
    if (feed != nullptr && CL > 1) {
      // A streamed launch follows the zeroing of its done counters in plain
      // stream order.
      cfg.attrs = attr + 1;
      cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, K::kernel, map_a, map_b, p) ==
                   cudaSuccess
               ? kOk
               : kErrLaunch;
  }
};

// The library's own stream-ordered memory pool on each device, for stream-K
// workspaces. Unlike the device's default pool (release threshold 0, which
// hands memory back to the driver at every synchronisation and makes the
// next allocation map it again), it keeps what it has reserved, so a
// workspace allocation after a synchronisation costs no more than one inside
// a busy stream.
int workspace_pool(int dev, cudaMemPool_t *out) {
  static cudaMemPool_t pools[64] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= 64) return kErrLaunch;
  std::lock_guard<std::mutex> g(mu);
  if (pools[dev] == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return kErrLaunch;
    uint64_t keep = ~0ull;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return kErrLaunch;
    }
    pools[dev] = pool;
  }
  *out = pools[dev];
  return kOk;
}

// Launch a prepared plan with its workspace (partial tiles, and counters
// cleared before the kernel) from the library's stream-ordered pool on the
// caller's stream, returned right after the kernel, so concurrent calls on
// other streams never share it.
template <class Plan>
int launch_pooled(Plan &plan, cudaStream_t stream) {
  void *ws = nullptr;
  if (plan.workspace_bytes() > 0) {
    int dev = 0;
    cudaMemPool_t pool = nullptr;
    if (cudaGetDevice(&dev) != cudaSuccess || workspace_pool(dev, &pool) != kOk) return kErrLaunch;
    if (cudaMallocFromPoolAsync(&ws, plan.workspace_bytes(), pool, stream) != cudaSuccess)
      return kErrLaunch;
    if (plan.counter_bytes > 0 && cudaMemsetAsync(ws, 0, plan.counter_bytes, stream) != cudaSuccess) {
      cudaFreeAsync(ws, stream);
      return kErrLaunch;
    }
    plan.set_workspace(ws);
  }
  const int st = plan.launch(stream);
  if (ws != nullptr && cudaFreeAsync(ws, stream) != cudaSuccess) return kErrLaunch;
  return st;
}

template <int BK, int STAGES, bool EXACT, bool LSU, int CL, bool OPB, bool OPA, int BST, bool PAIR,
          bool SCALED>
int launch_plans(const GemmArgs &a, int sm_count, cudaStream_t stream) {
  if constexpr (PAIR) {
    // Few unit tiles: pairs of one cluster share each tile.
    LaunchPlan<BK, STAGES, EXACT, LSU, CL, OPB, OPA, BST, PAIR, true, SCALED> cs;
    const int cst = cs.prepare(a, sm_count);
    if (cst != kOk) return cst;
    if (cs.p.ks > 1) return launch_pooled(cs, stream);
  }
  LaunchPlan<BK, STAGES, EXACT, LSU, CL, OPB, OPA, BST, PAIR, false, SCALED> plan;
  const int st = plan.prepare(a, sm_count);
  if (st != kOk) return st;
  return launch_pooled(plan, stream);
}

// The pair kernels come in two builds, for C = A B as it is and for
// alpha != 1 or beta != 0; the plain-load kernel handles both at run time.
template <int BK, int STAGES, bool EXACT, bool LSU, int CL, bool OPB, bool OPA = false,
          int BST = 0, bool PAIR = false>
int launch_variant(const GemmArgs &a, int sm_count, cudaStream_t stream) {
  if (PAIR && (a.alpha != 1.0f || a.beta != 0.0f))
    return launch_plans<BK, STAGES, EXACT, LSU, CL, OPB, OPA, BST, PAIR, PAIR>(a, sm_count, stream);
  return launch_plans<BK, STAGES, EXACT, LSU, CL, OPB, OPA, BST, PAIR, false>(a, sm_count, stream);
}

}  // namespace

int pool_alloc(void **ptr, size_t bytes, cudaStream_t stream) {
  int dev = 0;
  cudaMemPool_t pool = nullptr;
  if (cudaGetDevice(&dev) != cudaSuccess || workspace_pool(dev, &pool) != kOk) return kErrLaunch;
  return cudaMallocFromPoolAsync(ptr, bytes, pool, stream) == cudaSuccess ? kOk : kErrLaunch;
}

int pool_free(void *ptr, cudaStream_t stream) {
  return cudaFreeAsync(ptr, stream) == cudaSuccess ? kOk : kErrLaunch;
}

bool tc_tma_direct(const GemmArgs &a) {
  return !a.opa && reinterpret_cast<uintptr_t>(a.A) % 16 == 0 && a.lda % 4 == 0 &&
         reinterpret_cast<uintptr_t>(a.B) % 16 == 0 && a.ldb % 4 == 0;
}

namespace {

// Stages of the CTA-pair kernel: 32 KiB each (128 A rows and 128 B^T rows of
// 32 k per CTA). Timed at 4096^3 and 8192 x 11008 x 4096: 4 stages 0.73 /
// 0.89 of the peak, 5 0.78 / 0.89, 6 0.80 / 0.86-0.96, 7 0.79 / 0.85 (the
// pipeline waits on copies, not on free slots, from 6 on).
constexpr int kPairStages = 6;

// Rings of the 3xTF32 pair kernel, per CTA: A stages of BK k (hi and lo, 128
// rows: 32 KiB at BK = 32) and B slots (BK x 128: 16 KiB); TMEM holds 256
// accumulator columns and four B^T slots of 2 BK columns. Each k-block costs
// one hand-over between the CTAs, which sets the pace of short k-blocks: at
// 4096^3 BK = 16 took 0.64 ms (0.49 with two relay threads), BK = 32 with
// the B tile inside four 48 KiB stages 0.43 ms.
constexpr int kPairExactBK = 32;
constexpr int kPairExactStages = 6;
constexpr int kPairExactBSlots = 2;

bool tma_operand_ok(const float *ptr, int64_t ld) {
  return reinterpret_cast<uintptr_t>(ptr) % 16 == 0 && ld % 4 == 0;
}

// Single-pass TF32 through the CTA-pair kernel, which reads every operand
// layout by TMA. Operands whose base or pitch TMA cannot take are first
// copied, in the layout they have, into rows with 16-byte pitches.
int pair_launch(const GemmArgs &a, int sm_count, cudaStream_t stream) {
  const bool a_ok = tma_operand_ok(a.A, a.lda), b_ok = tma_operand_ok(a.B, a.ldb);
  if (!a_ok || !b_ok) {
    auto up4 = [](int64_t x) { return (x + 3) / 4 * 4; };
    auto up256 = [](size_t b) { return (b + 255) / 256 * 256; };
    const int64_t a_rows = a.opa ? a.K : a.M, a_cols = a.opa ? a.M : a.K;
    const int64_t b_rows = a.opb ? a.N : a.K, b_cols = a.opb ? a.K : a.N;
    const int64_t lda_p = up4(a_cols), ldb_p = up4(b_cols);
    const size_t a_bytes = a_ok ? 0 : up256(static_cast<size_t>(a_rows) * lda_p * 4);
    const size_t b_bytes = b_ok ? 0 : up256(static_cast<size_t>(b_rows) * ldb_p * 4);
    void *ws = nullptr;
    int st = pool_alloc(&ws, a_bytes + b_bytes, stream);
    if (st != kOk) return st;
    GemmArgs t = a;
    PackJob ja, jb;  // both copies in one launch
    if (!a_ok) {
      float *pa = static_cast<float *>(ws);
      ja = PackJob{a.A, a.lda, a_rows, a_cols, pa, lda_p};
      t.A = pa;
      t.lda = lda_p;
    }
    if (!b_ok) {
      float *pb = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + a_bytes);
      jb = PackJob{a.B, a.ldb, b_rows, b_cols, pb, ldb_p};
      t.B = pb;
      t.ldb = ldb_p;
    }
    st = pack_rows_launch(ja, jb, sm_count, stream);
    if (st == kOk) st = pair_launch(t, sm_count, stream);
    const int fst = pool_free(ws, stream);
    return st != kOk ? st : fst;
  }
  if (a.opa) {
    if (a.opb)
      return launch_variant<32, kPairStages, false, false, 2, true, true, 0, true>(a, sm_count,
                                                                                    stream);
    return launch_variant<32, kPairStages, false, false, 2, false, true, 0, true>(a, sm_count,
                                                                                   stream);
  }
  if (a.opb)
    return launch_variant<32, kPairStages, false, false, 2, true, false, 0, true>(a, sm_count,
                                                                                   stream);
  return launch_variant<32, kPairStages, false, false, 2, false, false, 0, true>(a, sm_count,
                                                                                  stream);
}

}  // namespace

int tc_launch(const GemmArgs &a, bool exact, bool lsu, int sm_count, cudaStream_t stream) {
  if (!exact && !lsu) return pair_launch(a, sm_count, stream);
  if (!lsu && !tc_tma_direct(a)) {
    // Operands TMA cannot describe as given: copy them into one workspace
    // from the library's pool with 16-byte row pitches (A stored transposed,
    // K x M, becomes a row-major M x K copy), ordered on the stream before
    // the GEMM and released after it.
    const bool a_ok = !a.opa && reinterpret_cast<uintptr_t>(a.A) % 16 == 0 && a.lda % 4 == 0;
    const bool b_ok = reinterpret_cast<uintptr_t>(a.B) % 16 == 0 && a.ldb % 4 == 0;
    auto up4 = [](int64_t x) { return (x + 3) / 4 * 4; };
    auto up256 = [](size_t b) { return (b + 255) / 256 * 256; };
    const int64_t b_rows = a.opb ? a.N : a.K, b_cols = a.opb ? a.K : a.N;
    const int64_t lda_p = up4(a.K), ldb_p = up4(b_cols);
    const size_t a_bytes = a_ok ? 0 : up256(static_cast<size_t>(a.M) * lda_p * 4);
    const size_t b_bytes = b_ok ? 0 : up256(static_cast<size_t>(b_rows) * ldb_p * 4);
    void *ws = nullptr;
    int st = pool_alloc(&ws, a_bytes + b_bytes, stream);
    if (st != kOk) return st;
    GemmArgs t = a;
    PackJob ja, jb;  // row copies of both operands in one launch
    if (!a_ok) {
      float *pa = static_cast<float *>(ws);
      if (a.opa)
        st = transpose_launch(a.A, a.lda, a.K, a.M, pa, lda_p, sm_count, stream);
      else
        ja = PackJob{a.A, a.lda, a.M, a.K, pa, lda_p};
      t.A = pa;
      t.lda = lda_p;
      t.opa = 0;
    }
    if (!b_ok) {
      float *pb = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + a_bytes);
      jb = PackJob{a.B, a.ldb, b_rows, b_cols, pb, ldb_p};
      t.B = pb;
      t.ldb = ldb_p;
    }
    if (st == kOk) st = pack_rows_launch(ja, jb, sm_count, stream);
    if (st == kOk) st = tc_launch(t, exact, false, sm_count, stream);
    const int fst = pool_free(ws, stream);
    return st != kOk ? st : fst;
  }
  if (a.opa) {
    // A stored transposed (K x M) for the LSU variant: the producer
    // transposes each tile on its way into shared memory; B as for A stored
    // row-major.
    if (a.opb) {
      if (exact) return launch_variant<16, 4, true, true, 1, true, true>(a, sm_count, stream);
      return launch_variant<32, 4, false, true, 1, true, true>(a, sm_count, stream);
    }
    if (exact) return launch_variant<16, 6, true, true, 1, false, true>(a, sm_count, stream);
    return launch_variant<32, 6, false, true, 1, false, true>(a, sm_count, stream);
  }
  if (a.opb) {
    // B stored transposed (N x K): its tile is K-major. The TMA-fed 3xTF32
    // pair kernel moves it into TMEM as B^T hi and lo, as for B stored K x N;
    // the LSU variants stage 48 KiB per stage (exact: A, B and their lo tiles
    // at BK = 16; tf32: A and B at 32).
    if (exact) {
      if (lsu) return launch_variant<16, 4, true, true, 1, true>(a, sm_count, stream);
      return launch_variant<kPairExactBK, kPairExactStages, true, false, 2, true, false,
                            kPairExactBSlots, true>(a, sm_count, stream);
    }
    return launch_variant<32, 4, false, true, 1, true>(a, sm_count, stream);
  }
  // B stored K x N. (One TF32 pass fed by TMA went to pair_launch above.)
  if (exact) {
    if (lsu) return launch_variant<16, 6, true, true, 1, false>(a, sm_count, stream);
    return launch_variant<kPairExactBK, kPairExactStages, true, false, 2, false, false,
                          kPairExactBSlots, true>(a, sm_count, stream);
  }
  return launch_variant<32, 6, false, true, 1, false>(a, sm_count, stream);
}

static_assert(kStreamRows == kTM, "a ready word and a done counter cover one row of unit tiles");
static_assert(kPairExactBK == kStreamKBlock, "B halves end on 3xTF32 pair k-blocks");

int tc_launch_streamed(const GemmArgs &a, const StreamFeed &feed, int sm_count,
                       cudaStream_t stream) {
  if (a.opa || a.opb || !tc_tma_direct(a) || a.K < 1) return kErrInvalidArg;
  LaunchPlan<kPairExactBK, kPairExactStages, true, false, 2, false, false, kPairExactBSlots, true>
      plan;
  plan.feed = &feed;
  const int st = plan.prepare(a, sm_count);
  return st != kOk ? st : plan.launch(stream);
}

GEMM_INDEX_FAULT_TAKE(tc_index_fault_take)

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

namespace {

// One launch of a TMA-fed pair kernel whose producers stop after their first
// k-block, with every wait limited to timeout_ns: the cluster-split variant
// when the problem takes it, else the plain one, which accepts only problems
// whose tiles are not split through a workspace.
template <class Plan>
int stalled_run(Plan &plan, int64_t timeout_ns, cudaStream_t stream) {
  plan.p.timeout_ns = static_cast<unsigned long long>(timeout_ns);
  plan.p.stall_kb = 1;
  const int st = launch_pooled(plan, stream);
  if (st != kOk) return st;
  return tc_poll_status(stream);
}

template <class CsPlan, class Plan>
int stalled_launch(const GemmArgs &a, int64_t timeout_ns, int sm_count, cudaStream_t stream) {
  CsPlan cs;
  int st = cs.prepare(a, sm_count);
  if (st != kOk) return st;
  if (cs.p.ks > 1) return stalled_run(cs, timeout_ns, stream);
  Plan plan;
  st = plan.prepare(a, sm_count);
  if (st != kOk) return st;
  if (plan.counter_bytes > 0) return kErrInvalidArg;
  return stalled_run(plan, timeout_ns, stream);
}

}  // namespace

int tc_selftest_stalled_gemm(const GemmArgs &a, bool exact, int64_t timeout_ns, int sm_count,
                             cudaStream_t stream) {
  if (!tc_tma_direct(a) || a.opb || a.K < 2 * 32) return kErrInvalidArg;
  if (exact)
    return stalled_launch<LaunchPlan<kPairExactBK, kPairExactStages, true, false, 2, false, false,
                                     kPairExactBSlots, true, true>,
                          LaunchPlan<kPairExactBK, kPairExactStages, true, false, 2, false, false,
                                     kPairExactBSlots, true>>(a, timeout_ns, sm_count, stream);
  return stalled_launch<LaunchPlan<32, kPairStages, false, false, 2, false, false, 0, true, true>,
                        LaunchPlan<32, kPairStages, false, false, 2, false, false, 0, true>>(
      a, timeout_ns, sm_count, stream);
}

}  // namespace gemm

// ------------------------------------------------- allocation-free variant --
//
// gemm_f32_noalloc runs the same tensor-core kernel as gemm_f32 but takes the
// stream-K workspace (split-tile partials and counters) from the fixed array
// below instead of the device's memory pool, for callers that must not
// allocate device memory while they run. The array is part of the library's
// device image: every GPU that loads the library keeps these bytes until the
// process exits, and all calls share them.

static __device__ __align__(256) unsigned char
    g_gemm_noalloc_scratch[GEMM_F32_NOALLOC_SCRATCH_BYTES];

namespace gemm {
namespace {

// Device address of the scratch array on each device. The host-side name of
// a __device__ array is only a stand-in for it, so the address is looked up
// once per device, with that device current.
struct NoAllocScratch {
  bool ready = false;
  void *ptr = nullptr;
};
NoAllocScratch g_noalloc[64];
std::mutex g_noalloc_mu;

int noalloc_scratch(int dev, void **out) {
  if (dev < 0 || dev >= 64) return kErrLaunch;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  NoAllocScratch &d = g_noalloc[dev];
  if (!d.ready) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gemm_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return kErrLaunch;
    d.ptr = ptr;
    d.ready = true;
  }
  *out = d.ptr;
  return kOk;
}

template <int BK, int STAGES, bool EXACT, bool LSU, int CL, bool OPB, int BST = 0,
          bool PAIR = false>
int launch_variant_noalloc(const GemmArgs &a, int sm_count, cudaStream_t stream) {
  // gemm_f32_noalloc computes C = A B: the pair kernels' unscaled build.
  if (a.alpha != 1.0f || a.beta != 0.0f) return kErrInvalidArg;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kErrLaunch;
  void *scratch = nullptr;
  int st = noalloc_scratch(dev, &scratch);
  if (st != kOk) return st;
  // The same workspace layout gemm_f32 takes from the pool, here inside the
  // fixed array; problems that need more are refused before anything runs.
  auto run_in_scratch = [&](auto &plan) {
    if (plan.workspace_bytes() > 0) {
      if (plan.workspace_bytes() > GEMM_F32_NOALLOC_SCRATCH_BYTES) return static_cast<int>(kErrInvalidArg);
      // The counters must start at zero; the previous call left them counted up.
      if (plan.counter_bytes > 0 && cudaMemsetAsync(scratch, 0, plan.counter_bytes, stream) != cudaSuccess)
        return static_cast<int>(kErrLaunch);
      plan.set_workspace(scratch);
    }
    return plan.launch(stream);
  };
  if constexpr (PAIR) {
    LaunchPlan<BK, STAGES, EXACT, LSU, CL, OPB, false, BST, PAIR, true> cs;
    st = cs.prepare(a, sm_count);
    if (st != kOk) return st;
    if (cs.p.ks > 1) return run_in_scratch(cs);
  }
  LaunchPlan<BK, STAGES, EXACT, LSU, CL, OPB, false, BST, PAIR> plan;
  st = plan.prepare(a, sm_count);
  if (st != kOk) return st;
  return run_in_scratch(plan);
}

}  // namespace

int tc_launch_noalloc(const GemmArgs &a, bool exact, bool lsu, int sm_count, cudaStream_t stream) {
  // Same kernels and stage shapes as tc_launch.
  if (exact) {
    if (lsu) return launch_variant_noalloc<16, 6, true, true, 1, false>(a, sm_count, stream);
    return launch_variant_noalloc<kPairExactBK, kPairExactStages, true, false, 2, false,
                                  kPairExactBSlots, true>(a, sm_count, stream);
  }
  if (lsu) return launch_variant_noalloc<32, 6, false, true, 1, false>(a, sm_count, stream);
  return launch_variant_noalloc<32, kPairStages, false, false, 2, false, 0, true>(a, sm_count,
                                                                                  stream);
}

}  // namespace gemm

// ------------------------------------------------- schedule self-check --
//
// gemm_f32_schedule_check: the stream-K partition of a launch, built and
// walked on the host with the kernels' own work-list code (UnitIter), and
// checked: every k-block of every unit tile covered exactly once, whole
// units spanning their tile's k range, a split tile's parts numbered 0 ..
// nparts - 1 in k order with the same part count, at most kMaxSplit parts,
// and partial-sum slots owned by their cluster and never shared.
extern "C" int gemm_f32_schedule_check(int64_t M, int64_t N, int64_t K, int64_t workers,
                                       int kernel_kind, int64_t *stats) {
  using namespace gemm;
  if (M < 1 || N < 1 || K < 1 || workers < 1 || workers > 4096 || kernel_kind < 0 ||
      kernel_kind > 3 || stats == nullptr || M >= (int64_t{1} << 31) || N >= (int64_t{1} << 31) ||
      K >= (int64_t{1} << 31))
    return GEMM_ERR_INVALID_ARG;
  // The launch shapes tc_launch uses: 3xTF32 and TF32 pairs, and the
  // plain-load kernel in 3xTF32 (BK 16) and TF32 (BK 32) mode.
  const bool pair = kernel_kind < 2, exact = kernel_kind == 0 || kernel_kind == 2;
  const int bk = kernel_kind == 0 ? kPairExactBK : (kernel_kind == 2 ? 16 : 32);
  TcParams p = {};
  set_tiles(p, M, N, K, bk, pair ? 2 : 1);
  p.group_m = kGroupM;
  p.ks = 1;
  p.sk_first = 0;
  const int64_t cells = static_cast<int64_t>(p.num_tiles) * p.num_k_blocks;
  if (cells > (int64_t{1} << 26)) return GEMM_ERR_INVALID_ARG;  // keep the check's memory small
  const int ks = pair ? cluster_split_ks(p.num_tiles, p.num_k_blocks, static_cast<int>(workers), bk,
                                         exact)
                      : 1;
  if (ks >= 2) {
    // Cluster split: pair c takes k-slice c % ks of unit tile c / ks; the
    // slices of a tile cover its k range once, in pair order, none empty.
    p.ks = ks;
    const int kb = p.num_k_blocks, pairs = p.num_tiles * ks;
    std::vector<int> next_kb(static_cast<size_t>(p.num_tiles), 0);
    for (int c = 0; c < pairs; ++c) {
      UnitIter it(p, c, pairs);
      WorkUnit u;
      if (!it.next(p, u)) return 23;  // a pair without work
      if (u.tile < 0 || u.tile >= p.num_tiles || u.kb0 >= u.kb1 || u.kb1 > kb) return 10;
      if (u.part != c % ks || u.nparts != ks) return 14;
      int &at = next_kb[static_cast<size_t>(u.tile)];
      if (u.kb0 != at) return at > u.kb0 ? 11 : 20;  // covered twice / k-block missed
      at = u.kb1;
      if (it.next(p, u) || !it.done(p)) return 19;  // more than one unit
    }
    for (int t = 0; t < p.num_tiles; ++t)
      if (next_kb[static_cast<size_t>(t)] != kb) return 20;
    stats[0] = p.num_tiles;
    stats[1] = kb;
    stats[2] = 0;
    stats[3] = 0;
    stats[4] = 0;
    stats[5] = 0;
    stats[6] = ks;
    stats[7] = pairs;
    stats[8] = ks;
    return GEMM_OK;
  }
  const Schedule sch = schedule_for(p, static_cast<int>(workers), bk, exact, pair);
  p.dp_tiles = sch.dp_tiles;
  p.sk_share = sch.sk_share;
  p.sk_ctas = sch.sk_ctas;
  p.sk_first = split_chunk_first(sch, static_cast<int>(workers), exact, pair) ? 1 : 0;
  const int kb = p.num_k_blocks, clusters = sch.grid;
  std::vector<int> cover(static_cast<size_t>(cells), 0);
  std::vector<int> part_owner(static_cast<size_t>(p.num_tiles) * kMaxSplit, -1);
  std::vector<int> part_kb0(static_cast<size_t>(p.num_tiles) * kMaxSplit, -1);
  std::vector<int> tile_parts(static_cast<size_t>(p.num_tiles), 0);
  std::vector<char> slot_used(static_cast<size_t>(2 * (p.sk_ctas > 0 ? p.sk_ctas : 1)), 0);
  int max_parts = 1;
  for (int c = 0; c < clusters; ++c) {
    UnitIter it(p, c, clusters);
    WorkUnit u;
    while (it.next(p, u)) {
      if (u.tile < 0 || u.tile >= p.num_tiles || u.kb0 < 0 || u.kb1 > kb || u.kb0 >= u.kb1)
        return 10;  // unit outside the problem
      for (int k = u.kb0; k < u.kb1; ++k)
        if (++cover[static_cast<size_t>(u.tile) * kb + k] > 1) return 11;  // covered twice
      if (u.nparts == 1) {
        if (u.kb0 != 0 || u.kb1 != kb) return 12;  // a whole unit must span the tile
        continue;
      }
      if (u.nparts < 1 || u.nparts > kMaxSplit) return 13;
      if (u.sk_tile != u.tile - p.dp_tiles || u.part < 0 || u.part >= u.nparts) return 14;
      if (u.slot < 0 || u.slot >= 2 * p.sk_ctas || u.slot / 2 != c) return 15;
      if (slot_used[static_cast<size_t>(u.slot)]++) return 16;  // slot shared
      const size_t t = static_cast<size_t>(u.tile) * kMaxSplit + u.part;
      if (part_owner[t] != -1) return 17;  // part index given twice
      part_owner[t] = c;
      part_kb0[t] = u.kb0;
      int &np = tile_parts[static_cast<size_t>(u.tile)];
      if (np != 0 && np != u.nparts) return 18;  // parts disagree on their count
      np = u.nparts;
      if (u.nparts > max_parts) max_parts = u.nparts;
    }
    if (!it.done(p)) return 19;
  }
  for (int64_t i = 0; i < cells; ++i)
    if (cover[static_cast<size_t>(i)] != 1) return 20;  // k-block missed
  for (int t = 0; t < p.num_tiles; ++t) {
    const int np = tile_parts[static_cast<size_t>(t)];
    for (int q = 0; q < np; ++q) {
      const size_t i = static_cast<size_t>(t) * kMaxSplit + q;
      if (part_owner[i] < 0) return 21;  // a part missing
      if (q > 0 && part_kb0[i] <= part_kb0[i - 1]) return 22;  // parts out of k order
    }
  }
  stats[0] = p.num_tiles;
  stats[1] = kb;
  stats[2] = p.dp_tiles;
  stats[3] = p.sk_share;
  stats[4] = p.sk_ctas;
  stats[5] = sch.splits ? 1 : 0;
  stats[6] = max_parts;
  stats[7] = clusters;
  stats[8] = 1;
  return GEMM_OK;
}
