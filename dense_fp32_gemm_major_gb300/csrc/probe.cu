// probe.cu -- what this GPU's pipes deliver with nothing else in the way:
// a TF32 tensor-core probe (tcgen05.mma kind::tf32 from resident shared
// memory into TMEM, no loads) and an FP32 FMA probe (independent FFMA chains
// in registers). The rates they measure are context for the roofline
// fractions, which stay against the measured bf16 peak; see bench.py.
//
// Both kernels run one CTA per SM. The tensor probe issues the same 128 x
// 256 x 8 MMA shape as the GEMM kernels, back to back on one accumulator,
// and waits (bounded) for their completion before freeing TMEM.

#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace gemm {

__device__ int g_probe_status;

namespace {

constexpr int kProbeSmem = 120 * 1024;  // > half an SM's shared memory: one CTA per SM
constexpr int kFmaChains = 8;

// Operands: a 128 x 32 tile and a 256 x 32 tile (K-major, 128-byte swizzle),
// zero (their values do not change the MMA's time).
__global__ void __launch_bounds__(128, 1) probe_tf32_kernel(int iters) {
  extern __shared__ uint8_t raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  for (int i = threadIdx.x; i < (128 + 256) * 32; i += blockDim.x)
    reinterpret_cast<float *>(tiles)[i] = 0.0f;
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
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_tf32(tmem, smem_desc(a + kk * 32, 16, 1024, 2), smem_desc(b + kk * 32, 16, 1024, 2),
                 idesc, (it | kk) ? 1u : 0u);
    }
    mma_commit(&done);
    mbar_wait_bounded(&done, 0, 4000000000ull, &abort_flag, &g_probe_status);
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
// chains are not removed.
__global__ void __launch_bounds__(1024, 1) probe_fma_kernel(int iters, float x, float *sink) {
  float acc[kFmaChains];
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) acc[c] = static_cast<float>(threadIdx.x + c);
  const float y = 1.0f - x;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kFmaChains; ++c) acc[c] = fmaf(acc[c], x, y);
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kFmaChains; ++c) s += acc[c];
  if (s == -1.0f) *sink = s;
}

}  // namespace

int probe_peaks(int sm_count, double *tf32_tflops, double *fp32_tflops, cudaStream_t stream) {
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
    return kErrLaunch;
  int st = kOk;
  float ms = 0.0f;
  // Tensor probe: iters x 4 MMAs of 2 * 128 * 256 * 8 flops per SM.
  const int mma_iters = 200000;
  if (cudaFuncSetAttribute(probe_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kProbeSmem) != cudaSuccess)
    st = kErrLaunch;
  for (int rep = 0; st == kOk && rep < 2; ++rep) {  // the first launch warms up
    cudaEventRecord(e0, stream);
    probe_tf32_kernel<<<sm_count, 128, kProbeSmem, stream>>>(mma_iters);
    cudaEventRecord(e1, stream);
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      st = kErrLaunch;
  }
  if (st == kOk) {
    const double flops = static_cast<double>(sm_count) * mma_iters * 4 * 2.0 * 128 * 256 * 8;
    *tf32_tflops = flops / (ms * 1e-3) / 1e12;
  }
  // FMA probe: 1024 threads per SM, kFmaChains chains of fma_iters FFMAs.
  const int fma_iters = 100000;
  float *sink = nullptr;
  if (st == kOk && cudaMalloc(&sink, sizeof(float)) != cudaSuccess) st = kErrLaunch;
  for (int rep = 0; st == kOk && rep < 2; ++rep) {
    cudaEventRecord(e0, stream);
    probe_fma_kernel<<<sm_count, 1024, 0, stream>>>(fma_iters, 0.999f, sink);
    cudaEventRecord(e1, stream);
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      st = kErrLaunch;
  }
  if (st == kOk) {
    const double flops = static_cast<double>(sm_count) * 1024 * fma_iters * kFmaChains * 2.0;
    *fp32_tflops = flops / (ms * 1e-3) / 1e12;
  }
  if (sink) cudaFree(sink);
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
