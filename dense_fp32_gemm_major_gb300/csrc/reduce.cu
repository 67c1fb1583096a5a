// reduce.cu -- sum of a fp32 vector: per-group partial sums, then a second
// dispatch that combines them.
//
// The reduction of "GPU compute shaders" ("How it works", step 6; the reduce
// routine under "Code"): every group walks the vector with a grid stride,
// reduces its invocations' sums by a tree in shared memory and writes one
// partial; a second dispatch sums the partials. For a fixed group count the
// order of every addition is fixed, so reruns are bit-identical (the page's
// "Pitfalls").
//
// On sm_103a the sum is bound by HBM bandwidth: each byte is read once. A
// group is a 256-thread CTA; the default grid is four CTAs per SM. Each
// thread keeps four independent fp32 accumulators (the components of its
// 128-bit loads) and has four 128-bit loads in flight, 16 KiB per CTA, which
// covers the memory latency at full bandwidth. The tree runs on warp shuffles
// (5 levels) and one shared-memory step across the 8 warps. The second
// dispatch is a programmatic dependent launch, so its start-up overlaps the
// first grid's tail.
//
// Error: every element reaches the result through at most
// h = ceil(n / (4 * 256 * G)) + ceil(G / 256) + 24 roundings (its
// accumulator's chain, the tail element, 2 to combine the four accumulators,
// 8 tree levels, the second dispatch's chain and its 8 tree levels), so
// |sum - exact| <= h * 2^-24 * sum |x| (to first order).

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace gemm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;  // the same value in every lane (each pair adds the same two terms)
}

// Sum of v over the CTA, valid in thread 0.
__device__ __forceinline__ float block_sum(float v) {
  __shared__ float warp_part[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) warp_part[warp] = v;
  __syncthreads();
  float w = 0.0f;
  if (warp == 0) {
    w = lane < kWarps ? warp_part[lane] : 0.0f;
#pragma unroll
    for (int m = kWarps / 2; m > 0; m >>= 1) w += __shfl_xor_sync(0xffffffffu, w, m);
  }
  return w;
}

// Group g = blockIdx.x writes partials[g]: the sum of the elements it visits.
// VEC: x is 16-byte aligned; float4 j goes to thread j mod T (T threads in
// all) and the n mod 4 tail elements to threads 0, 1, 2. Otherwise element
// i goes to thread i mod T.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    reduce_partials_kernel(const float *__restrict__ x, long long n, float *__restrict__ partials,
                           int groups) {
  // Let the second dispatch be scheduled now; it waits for this grid to
  // finish (and its writes to land) before it reads the partials.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long T = static_cast<long long>(gridDim.x) * kThreads;
  const long long t = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  if (VEC) {
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const long long n4 = n >> 2;
    long long i = t;
    for (; i + (kUnroll - 1) * T < n4; i += kUnroll * T) {
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        v[u] = index_ok(kSiteReduceIn, 4 * (i + u * T), 4, n) ? __ldcs(x4 + i + u * T)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        a0 += v[u].x;
        a1 += v[u].y;
        a2 += v[u].z;
        a3 += v[u].w;
      }
    }
    for (; i < n4; i += T) {
      const float4 v = index_ok(kSiteReduceIn, 4 * i, 4, n) ? __ldcs(x4 + i)
                                                            : make_float4(0.f, 0.f, 0.f, 0.f);
      a0 += v.x;
      a1 += v.y;
      a2 += v.z;
      a3 += v.w;
    }
    if (t < n - 4 * n4 && index_ok(kSiteReduceIn, 4 * n4 + t, 1, n)) a0 += x[4 * n4 + t];
  } else {
    long long i = t;
    auto load = [&](long long j) {
      return index_ok(kSiteReduceIn, j, 1, n) ? __ldcs(x + j) : 0.0f;
    };
    for (; i + 3 * T < n; i += 4 * T) {
      const float v0 = load(i), v1 = load(i + T), v2 = load(i + 2 * T), v3 = load(i + 3 * T);
      a0 += v0;
      a1 += v1;
      a2 += v2;
      a3 += v3;
    }
    for (; i < n; i += T) a0 += load(i);
  }
  const float s = block_sum((a0 + a1) + (a2 + a3));
  if (threadIdx.x == 0 && index_ok(kSiteReducePartial, blockIdx.x, 1, groups))
    partials[blockIdx.x] = s;
}

// The second dispatch: one CTA sums the G partials (partial g to thread
// g mod 256, then the tree) into *out.
__global__ void __launch_bounds__(kThreads)
    reduce_final_kernel(const float *__restrict__ partials, int groups, float *__restrict__ out) {
  // Launched as a programmatic dependent of the partial-sum grid: wait until
  // that grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float a = 0.0f;
  for (int g = threadIdx.x; g < groups; g += kThreads)
    if (index_ok(kSiteReducePartial, g, 1, groups)) a += partials[g];
  const float s = block_sum(a);
  if (threadIdx.x == 0) *out = s;
}

}  // namespace

GEMM_INDEX_FAULT_TAKE(reduce_index_fault_take)

int reduce_default_groups(int sm_count) { return 4 * (sm_count > 0 ? sm_count : 1); }

int reduce_launch(int64_t n, const float *x, float *out, int groups, float *partials,
                  cudaStream_t stream) {
  if (n == 0) {
    return cudaMemsetAsync(out, 0, sizeof(float), stream) == cudaSuccess ? kOk : kErrLaunch;
  }
  if (reinterpret_cast<uintptr_t>(x) % 16 == 0)
    reduce_partials_kernel<true><<<groups, kThreads, 0, stream>>>(x, n, partials, groups);
  else
    reduce_partials_kernel<false><<<groups, kThreads, 0, stream>>>(x, n, partials, groups);
  if (cudaGetLastError() != cudaSuccess) return kErrLaunch;
  // The second dispatch as a programmatic dependent launch: its launch
  // overlaps the tail of the first grid instead of following its completion.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reduce_final_kernel, static_cast<const float *>(partials),
                            groups, out) == cudaSuccess
             ? kOk
             : kErrLaunch;
}

}  // namespace gemm
