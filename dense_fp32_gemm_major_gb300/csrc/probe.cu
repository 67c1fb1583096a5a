// probe.cu -- what this GPU's pipes deliver with nothing else in the way:
// a TF32 tensor-core probe (tcgen05.mma kind::tf32 from resident shared
// memory into TMEM, no loads) and an FP32 FMA probe (independent FFMA chains
// in registers). The rates they measure are context for the roofline
// fractions, which stay against the measured bf16 peak; see bench.py.
//
// Both kernels run one CTA per SM. The tensor probe issues the same 128 x
// 256 x 8 MMA shape as the GEMM kernels, back to back on one accumulator,
// from operand tiles filled with non-zero values (a pipe multiplying zeros
// may draw less power, and so hold a higher clock under a power cap, than one
// multiplying data), and waits (bounded) for their completion before freeing
// TMEM. Each CTA also records the SM clock ticks (clock64) and the wall time
// (%globaltimer, ns) its timed part took, so the host can state the SM clock
// each rate was measured at.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "kernels.h"
#include "ptx.cuh"

namespace gemm {

__device__ int g_probe_status;

namespace {

constexpr int kProbeSmem = 120 * 1024;  // > half an SM's shared memory: one CTA per SM
constexpr int kFmaChains = 8;

// Operand value for element i: an integer hash of (seed, i) (multiply by
// Knuth's 2654435761, then xor-shift) mapped onto [-1, 1) in steps of 2^-23.
__device__ __forceinline__ float probe_value(uint32_t seed, uint32_t i) {
  uint32_t h = (i + 1u) * 2654435761u ^ seed;
  h ^= h >> 15;
  h *= 2654435761u;
  h ^= h >> 13;
  return static_cast<float>(static_cast<int32_t>(h >> 8) - (1 << 23)) * (1.0f / 8388608.0f);
}

// Operands: a 128 x 32 tile and a 256 x 32 tile (K-major, 128-byte swizzle),
// filled with probe_value. clocks[2 b], clocks[2 b + 1]: SM clock ticks and
// ns from the first MMA issued by CTA b to the completion of its last.
__global__ void __launch_bounds__(128, 1) probe_tf32_kernel(int iters, uint32_t seed,
                                                            unsigned long long *clocks) {
  extern __shared__ uint8_t raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  for (int i = threadIdx.x; i < (128 + 256) * 32; i += blockDim.x)
    reinterpret_cast<float *>(tiles)[i] = probe_value(seed, static_cast<uint32_t>(i));
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;
  if (threadIdx.x == 0) {
    const uint32_t a = smem_addr(tiles), b = smem_addr(tiles + 128 * 128);
    const uint32_t idesc = idesc_tf32(128, 256);
    const unsigned long long c0 = clock64();
    const uint64_t t0 = global_timer_ns();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_tf32(tmem, smem_desc(a + kk * 32, 16, 1024, 2), smem_desc(b + kk * 32, 16, 1024, 2),
                 idesc, (it | kk) ? 1u : 0u);
    }
    mma_commit(&done);
    mbar_wait_bounded(&done, 0, 4000000000ull, &abort_flag, &g_probe_status);
    clocks[2 * blockIdx.x] = clock64() - c0;
    clocks[2 * blockIdx.x + 1] = global_timer_ns() - t0;
  }
  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

// kFmaChains independent multiply-add chains per thread; the result is
// stored (conditionally on a value the host never passes) so that the
// chains are not removed. Thread 0 of CTA b records the SM clock ticks and ns
// its chains took in clocks[2 b], clocks[2 b + 1].
__global__ void __launch_bounds__(1024, 1) probe_fma_kernel(int iters, float x, float *sink,
                                                            unsigned long long *clocks) {
  float acc[kFmaChains];
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) acc[c] = static_cast<float>(threadIdx.x + c);
  const float y = 1.0f - x;
  const unsigned long long c0 = clock64();
  const uint64_t t0 = global_timer_ns();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) acc[c] = fmaf(acc[c], x, y);
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) s += acc[c];
  if (s == -1.0f) *sink = s;
  if (threadIdx.x == 0) {
    clocks[2 * blockIdx.x] = clock64() - c0;
    clocks[2 * blockIdx.x + 1] = global_timer_ns() - t0;
  }
}

// Median over the CTAs of ticks / ns, in MHz.
double median_mhz(const std::vector<unsigned long long> &clocks) {
  std::vector<double> mhz;
  for (size_t b = 0; b + 1 < clocks.size(); b += 2)
    if (clocks[b + 1] > 0) mhz.push_back(1e3 * static_cast<double>(clocks[b]) / clocks[b + 1]);
  if (mhz.empty()) return 0.0;
  std::sort(mhz.begin(), mhz.end());
  return mhz[mhz.size() / 2];
}

}  // namespace

int probe_peaks(int sm_count, double *tf32_tflops, double *fp32_tflops, double *tf32_mhz,
                double *fp32_mhz, cudaStream_t stream) {
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
    return kErrLaunch;
  int st = kOk;
  float ms = 0.0f;
  float *sink = nullptr;
  unsigned long long *clocks = nullptr;
  std::vector<unsigned long long> host(2 * static_cast<size_t>(sm_count));
  const size_t clock_bytes = host.size() * sizeof(unsigned long long);
  if (cudaMalloc(&sink, sizeof(float)) != cudaSuccess ||
      cudaMalloc(&clocks, clock_bytes) != cudaSuccess)
    st = kErrLaunch;
  // Tensor probe: iters x 4 MMAs of 2 * 128 * 256 * 8 flops per SM.
  const int mma_iters = 200000;
  if (st == kOk && cudaFuncSetAttribute(probe_tf32_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kProbeSmem) != cudaSuccess)
    st = kErrLaunch;
  for (int rep = 0; st == kOk && rep < 2; ++rep) {  // the first launch warms up
    cudaEventRecord(e0, stream);
    probe_tf32_kernel<<<sm_count, 128, kProbeSmem, stream>>>(mma_iters, 0x5eedu + rep, clocks);
    cudaEventRecord(e1, stream);
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      st = kErrLaunch;
  }
  if (st == kOk && cudaMemcpy(host.data(), clocks, clock_bytes, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
    st = kErrLaunch;
  if (st == kOk) {
    const double flops = static_cast<double>(sm_count) * mma_iters * 4 * 2.0 * 128 * 256 * 8;
    *tf32_tflops = flops / (ms * 1e-3) / 1e12;
    *tf32_mhz = median_mhz(host);
  }
  // FMA probe: 1024 threads per SM, kFmaChains chains of fma_iters FFMAs.
  const int fma_iters = 100000;
  for (int rep = 0; st == kOk && rep < 2; ++rep) {
    cudaEventRecord(e0, stream);
    probe_fma_kernel<<<sm_count, 1024, 0, stream>>>(fma_iters, 0.999f, sink, clocks);
    cudaEventRecord(e1, stream);
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      st = kErrLaunch;
  }
  if (st == kOk && cudaMemcpy(host.data(), clocks, clock_bytes, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
    st = kErrLaunch;
  if (st == kOk) {
    const double flops = static_cast<double>(sm_count) * 1024 * fma_iters * kFmaChains * 2.0;
    *fp32_tflops = flops / (ms * 1e-3) / 1e12;
    *fp32_mhz = median_mhz(host);
  }
  if (sink) cudaFree(sink);
  if (clocks) cudaFree(clocks);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st == kOk) {
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_probe_status, sizeof(int)) != cudaSuccess) return kErrLaunch;
    if (h != 0) return h;
  }
  return st;
}

}  // namespace gemm
