// api.cu -- the C ABI of libgemm_f32.so (declared in include/gemm_f32.h):
// argument validation, kernel selection and launch, the host-buffer entry
// point and status reporting.
//
// The interface follows the dispatch routine of "WebGPU WGSL Compute Shaders:
// Custom Matrix Multiplication (GEMM) Optimization Guide", section 5
// (executeGemm(device, M, N, K, bufA, bufB, bufC): caller-owned buffers,
// sizes passed at run time, asynchronous submission), with leading
// dimensions, an accuracy mode, a stream and a returned status added.

#include <cuda.h>
#include <cuda_runtime.h>

#include <chrono>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <thread>

#include "../../include/gemm_f32.h"
#include "../../include/reduce_f32.h"
#include "kernels.h"

namespace {

using gemm::GemmArgs;

constexpr int64_t kMaxDim = 0x7fffffffLL;  // sizes and leading dimensions < 2^31
constexpr int64_t kMaxSpan = int64_t{1} << 44;  // elements one matrix may span

struct DeviceInfo {
  bool probed = false;
  bool supported = false;
  int sm_count = 0;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Capability check and SM count for the current device (cached).
int current_device(int *dev_out, int *sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return gemm::kErrLaunch;
  if (dev < 0 || dev >= kMaxDevices) return gemm::kErrUnsupportedDevice;
  std::lock_guard<std::mutex> g(g_devices_mu);
  DeviceInfo &d = g_devices[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return gemm::kErrLaunch;
    d.supported = (major == 10 && minor == 3);
    d.sm_count = sms;
    d.probed = true;
  }
  if (!d.supported) return gemm::kErrUnsupportedDevice;
  *dev_out = dev;
  *sm_count = d.sm_count;
  return gemm::kOk;
}

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
  return a0 < b1 && b0 < a1;
}

// Elements spanned by a rows x cols row-major matrix with pitch ld. With
// every argument in [1, 2^31) the product stays below 2^62.
int64_t matrix_span(int64_t rows, int64_t cols, int64_t ld) { return (rows - 1) * ld + cols; }

// Byte range [lo, hi) touched by a rows x cols row-major matrix with pitch ld
// (its span checked against kMaxSpan first, so the byte count cannot wrap).
void matrix_range(const void *p, int64_t rows, int64_t cols, int64_t ld, uintptr_t *lo,
                  uintptr_t *hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + static_cast<uintptr_t>(matrix_span(rows, cols, ld)) * 4;
}

// Host-only validation. Returns kOk, or an error; *noop is set when there is
// nothing to compute (M == 0 or N == 0).
int validate(const GemmArgs &a, int mode, bool *noop) {
  *noop = false;
  if (mode != GEMM_F32_EXACT && mode != GEMM_F32_TF32 && mode != GEMM_F32_EXACT_SIMT)
    return gemm::kErrInvalidArg;
  if ((a.opa != GEMM_OP_N && a.opa != GEMM_OP_T) || (a.opb != GEMM_OP_N && a.opb != GEMM_OP_T))
    return gemm::kErrInvalidArg;
  if (a.M < 0 || a.N < 0 || a.K < 0) return gemm::kErrInvalidArg;
  if (a.M > kMaxDim || a.N > kMaxDim || a.K > kMaxDim) return gemm::kErrInvalidArg;
  // A is M x K (op N) or stored transposed, K x M (op T); B is K x N or N x K.
  const int64_t a_rows = a.opa ? a.K : a.M, a_cols = a.opa ? a.M : a.K;
  const int64_t b_rows = a.opb ? a.N : a.K, b_cols = a.opb ? a.K : a.N;
  if (a.lda < (a_cols > 1 ? a_cols : 1) || a.ldb < (b_cols > 1 ? b_cols : 1) ||
      a.ldc < (a.N > 1 ? a.N : 1))
    return gemm::kErrInvalidArg;
  if (a.lda > kMaxDim || a.ldb > kMaxDim || a.ldc > kMaxDim) return gemm::kErrInvalidArg;
  if (a.M == 0 || a.N == 0) {
    *noop = true;
    return gemm::kOk;
  }
  if (a.C == nullptr || reinterpret_cast<uintptr_t>(a.C) % 4 != 0) return gemm::kErrInvalidArg;
  if (matrix_span(a.M, a.N, a.ldc) > kMaxSpan) return gemm::kErrInvalidArg;
  if (a.K > 0) {
    if (a.A == nullptr || a.B == nullptr) return gemm::kErrInvalidArg;
    if (matrix_span(a_rows, a_cols, a.lda) > kMaxSpan ||
        matrix_span(b_rows, b_cols, a.ldb) > kMaxSpan)
      return gemm::kErrInvalidArg;
    if (reinterpret_cast<uintptr_t>(a.A) % 4 != 0 || reinterpret_cast<uintptr_t>(a.B) % 4 != 0)
      return gemm::kErrInvalidArg;
    uintptr_t c0, c1, x0, x1;
    matrix_range(a.C, a.M, a.N, a.ldc, &c0, &c1);
    matrix_range(a.A, a_rows, a_cols, a.lda, &x0, &x1);
    if (ranges_overlap(c0, c1, x0, x1)) return gemm::kErrAlias;
    matrix_range(a.B, b_rows, b_cols, a.ldb, &x0, &x1);
    if (ranges_overlap(c0, c1, x0, x1)) return gemm::kErrAlias;
  }
  return gemm::kOk;
}

// Kernel for (validated, non-empty) arguments, or -kErrInvalidArg. With
// can_pack the TMA-fed kernel serves any operands (those TMA cannot describe
// are copied into a workspace first); without it (no allocation allowed)
// only operands it can read as given.
int select_kernel(const GemmArgs &a, int mode, int kernel, bool can_pack = true) {
  const bool tma_ok = can_pack || gemm::tc_tma_direct(a);
  switch (kernel) {
    case GEMM_KERNEL_AUTO:
      if (mode == GEMM_F32_EXACT_SIMT) return GEMM_KERNEL_SIMT;
      // 3xTF32 keeps a per-product error near 2^-21 independent of K, which
      // fits the FP32-class bound 2 K 2^-24 only from K of about 8 on; below
      // 16 the exact mode takes the FP32 FMA kernel.
      if (mode == GEMM_F32_EXACT && a.K < 16) return GEMM_KERNEL_SIMT;
      return tma_ok ? GEMM_KERNEL_TC_TMA : GEMM_KERNEL_TC_LSU;
    case GEMM_KERNEL_SIMT:
      return mode == GEMM_F32_TF32 ? -gemm::kErrInvalidArg : GEMM_KERNEL_SIMT;
    case GEMM_KERNEL_TC_TMA:
      if (mode == GEMM_F32_EXACT_SIMT || !tma_ok) return -gemm::kErrInvalidArg;
      return GEMM_KERNEL_TC_TMA;
    case GEMM_KERNEL_TC_LSU:
      if (mode == GEMM_F32_EXACT_SIMT) return -gemm::kErrInvalidArg;
      return GEMM_KERNEL_TC_LSU;
    default:
      return -gemm::kErrInvalidArg;
  }
}

int run(const GemmArgs &a, int mode, int kernel, cudaStream_t stream) {
  bool noop = false;
  int st = validate(a, mode, &noop);
  if (st != gemm::kOk || noop) return st;
  const int k = select_kernel(a, mode, kernel);
  if (k < 0) return -k;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  if (a.K == 0 || a.alpha == 0.0f) {
    // No product term: C = beta * C, and C = 0 when beta == 0 (C not read).
    if (a.beta == 0.0f) {
      if (cudaMemset2DAsync(a.C, static_cast<size_t>(a.ldc) * 4, 0, static_cast<size_t>(a.N) * 4,
                            static_cast<size_t>(a.M), stream) != cudaSuccess)
        return gemm::kErrLaunch;
      return gemm::kOk;
    }
    // The FP32 kernel over an empty k range stores 0 * 0 + beta * C.
    GemmArgs s = a;
    s.K = 0;
    s.alpha = 0.0f;
    return gemm::simt_launch(s, sms, true, stream);
  }
  switch (k) {
    case GEMM_KERNEL_SIMT:
      return gemm::simt_launch(a, sms, true, stream);
    case GEMM_KERNEL_TC_TMA:
      return gemm::tc_launch(a, mode == GEMM_F32_EXACT, /*lsu=*/false, sms, stream);
    default:
      return gemm::tc_launch(a, mode == GEMM_F32_EXACT, /*lsu=*/true, sms, stream);
  }
}

// Per-device state of gemm_f32_host: a compute stream, one stream per copy
// direction, the events that chain row chunks through them, and grow-only
// device buffers.
constexpr int kHostMaxChunks = 16;
struct HostState {
  std::mutex mu;
  cudaStream_t stream = nullptr, h2d = nullptr, d2h = nullptr;
  cudaEvent_t a_in[kHostMaxChunks] = {}, c_done[kHostMaxChunks] = {}, b_hi = nullptr;
  cudaEvent_t cleared = nullptr;  // streamed calls: the done counters are zeroed
  bool ready = false;
  float *buf = nullptr;
  size_t cap_bytes = 0;
  // Streamed calls: words[0, cap) ready words of A's rows of unit tiles,
  // words[cap, cap + 2) of B's halves, words[cap + 2, 2 cap + 2) done
  // counters of C's rows (layout fixed per allocation, zeroed when made, so
  // a ready word only ever holds an earlier call's epoch).
  unsigned *words = nullptr;
  int64_t words_cap = 0;
  unsigned epoch = 0;
};
HostState g_host[kMaxDevices];

int host_state_init(HostState &hs) {
  if (hs.ready) return gemm::kOk;
  if (cudaStreamCreateWithFlags(&hs.stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hs.h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hs.d2h, cudaStreamNonBlocking) != cudaSuccess)
    return gemm::kErrLaunch;
  for (int i = 0; i < kHostMaxChunks; ++i)
    if (cudaEventCreateWithFlags(&hs.a_in[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hs.c_done[i], cudaEventDisableTiming) != cudaSuccess)
      return gemm::kErrLaunch;
  if (cudaEventCreateWithFlags(&hs.b_hi, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&hs.cleared, cudaEventDisableTiming) != cudaSuccess)
    return gemm::kErrLaunch;
  hs.ready = true;
  return gemm::kOk;
}

int64_t round_up4(int64_t x) { return (x + 3) / 4 * 4; }

// Stream memory operations of the driver (cuStreamWriteValue32: write a word
// once the stream's earlier work has completed; cuStreamWaitValue32: hold the
// stream until a word satisfies a condition). Looked up at run time, like the
// tensor-map encoder, so the library does not link libcuda. Null if the
// driver does not offer them.
typedef CUresult (*StreamValueFn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
struct StreamValueOps {
  StreamValueFn write = nullptr, wait = nullptr;
};
const StreamValueOps &stream_value_ops() {
  static StreamValueOps ops;
  static std::once_flag once;
  std::call_once(once, [] {
    void *w = nullptr, *v = nullptr;
    cudaDriverEntryPointQueryResult qw, qv;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &w, 12000, cudaEnableDefault,
                                         &qw) == cudaSuccess &&
        qw == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuStreamWaitValue32", &v, 12000, cudaEnableDefault,
                                         &qv) == cudaSuccess &&
        qv == cudaDriverEntryPointSuccess) {
      ops.write = reinterpret_cast<StreamValueFn>(w);
      ops.wait = reinterpret_cast<StreamValueFn>(v);
    }
  });
  return ops;
}

// gemm_f32_host in exact mode: one persistent 3xTF32 GEMM launch fed
// while it runs. The copy stream sends B's first half of k (all of B when K
// < 512), then A in blocks of up to 1024 rows, B's second half after the
// first block(s), writing one ready word after each; the kernel's
// producers wait (bounded) for the words of what they copy next. Its
// epilogue counts the stored tiles of each block, and the return stream
// copies each block of C to the host as soon as its count is complete. One
// launch over all tiles instead of one per row chunk. Copies stay large and
// words few: each word written after a copy waits for that copy to drain
// (about 3.5 us, and the next copy starts behind it), and 4 MiB copies moved
// 192 GB/s against 209 for one of 64 MiB.
// Self-test only: skip_block >= 0 leaves that block's ready word unwritten
// and timeout_ns > 0 limits each of the kernel's waits (see
// gemm_f32_selftest_host_missing_block).
int host_streamed(HostState &hs, const GemmArgs &host, int sms, float *dA, int64_t dlda,
                  float *dB, int64_t dldb, float *dC, int64_t dldc, int64_t skip_block = -1,
                  unsigned long long timeout_ns = 0) {
  const StreamValueOps &ops = stream_value_ops();
  const int64_t M = host.M, N = host.N, K = host.K;
  const int64_t rows = gemm::kStreamRows;
  const int64_t tiles_m = (M + rows - 1) / rows;  // rows of unit tiles
  // Rows of unit tiles per copy (and per word): a quarter of them, 1 to 4
  // (256 to 1024 rows of A and of C).
  int64_t per_copy = (tiles_m + 3) / 4;
  if (per_copy > 4) per_copy = 4;
  if (per_copy < 1) per_copy = 1;
  const int64_t tr = (tiles_m + per_copy - 1) / per_copy;  // copies of A, and of C
  // Rows of unit tiles [g0, g1) of copy i.
  auto group_rows = [&](int64_t i, int64_t &g0, int64_t &g1) {
    g0 = i * per_copy;
    g1 = g0 + per_copy < tiles_m ? g0 + per_copy : tiles_m;
  };
  if (tr > hs.words_cap) {
    if (hs.words) cudaFree(hs.words);
    hs.words = nullptr;
    hs.words_cap = 0;
    const size_t bytes = static_cast<size_t>(2 * tr + 2) * 4;
    if (cudaMalloc(&hs.words, bytes) != cudaSuccess) return gemm::kErrLaunch;
    if (cudaMemset(hs.words, 0, bytes) != cudaSuccess) return gemm::kErrLaunch;
    hs.words_cap = tr;
    hs.epoch = 0;
  }
  if (++hs.epoch == 0) {  // wrapped: clear the words so no old epoch can match
    if (cudaMemset(hs.words, 0, static_cast<size_t>(2 * hs.words_cap + 2) * 4) != cudaSuccess)
      return gemm::kErrLaunch;
    hs.epoch = 1;
  }
  const unsigned epoch = hs.epoch;
  unsigned *a_ready = hs.words, *b_ready = hs.words + hs.words_cap;
  unsigned *c_done = hs.words + hs.words_cap + 2;
  auto dptr = [](const void *p) { return static_cast<CUdeviceptr>(reinterpret_cast<uintptr_t>(p)); };

  // B's halves: rows [0, k1) and [k1, K), k1 a multiple of the k-block; all
  // of B in the first when K < 512.
  const int64_t kblk = gemm::kStreamKBlock;
  const int64_t k1 = K >= 512 ? (K / 2) / kblk * kblk : K;
  // Copies of A sent before B's second half: enough rows for a unit tile
  // per CTA pair, and no more bytes than that half of B, at least one.
  const int64_t nu = (N + 255) / 256;
  int64_t lead_rows = (sms / 2 + nu - 1) / nu;
  const int64_t half_b_rows = ((K - k1) * N) / (rows * K) + 1;
  if (lead_rows > half_b_rows) lead_rows = half_b_rows;
  int64_t lead = lead_rows / per_copy;
  if (lead < 1) lead = 1;

  auto drain = [&hs](int code) {
    cudaStreamSynchronize(hs.h2d);
    cudaStreamSynchronize(hs.stream);
    cudaStreamSynchronize(hs.d2h);
    return code;
  };
  // The done counters are zeroed on the compute stream before the kernel;
  // the return stream waits for that before it watches them.
  if (cudaMemsetAsync(c_done, 0, static_cast<size_t>(tr) * 4, hs.stream) != cudaSuccess ||
      cudaEventRecord(hs.cleared, hs.stream) != cudaSuccess)
    return drain(gemm::kErrLaunch);
  gemm::StreamFeed feed;
  feed.a_ready = a_ready;
  feed.b_ready = b_ready;
  feed.c_done = c_done;
  feed.epoch = epoch;
  feed.kb_split = static_cast<int>((k1 + kblk - 1) / kblk);
  feed.group = static_cast<int>(per_copy);
  feed.timeout_ns = timeout_ns;
  const GemmArgs d{M, N, K, dA, dlda, dB, dldb, dC, dldc};
  int st = gemm::tc_launch_streamed(d, feed, sms, hs.stream);
  if (st != gemm::kOk) return drain(st);

  // Inputs, each followed by its ready word.
  auto ready = [&](const unsigned *w) {
    return ops.write(hs.h2d, dptr(w), epoch, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
  };
  auto copy_b = [&](int64_t r0, int64_t n) {
    return cudaMemcpy2DAsync(dB + r0 * dldb, dldb * 4, host.B + r0 * host.ldb, host.ldb * 4,
                             N * 4, n, cudaMemcpyHostToDevice, hs.h2d) == cudaSuccess;
  };
  if (!copy_b(0, k1) || !ready(b_ready)) return drain(gemm::kErrLaunch);
  for (int64_t i = 0; i < tr; ++i) {
    int64_t b0, b1;
    group_rows(i, b0, b1);
    const int64_t r0 = b0 * rows, n = (b1 * rows < M ? b1 * rows : M) - r0;
    if (cudaMemcpy2DAsync(dA + r0 * dlda, dlda * 4, host.A + r0 * host.lda, host.lda * 4, K * 4,
                          n, cudaMemcpyHostToDevice, hs.h2d) != cudaSuccess ||
        (i != skip_block && !ready(a_ready + i)))
      return drain(gemm::kErrLaunch);
    if (i + 1 == lead && k1 < K && (!copy_b(k1, K - k1) || !ready(b_ready + 1)))
      return drain(gemm::kErrLaunch);
  }
  // Outputs: each block of C once its tiles are stored.
  if (cudaStreamWaitEvent(hs.d2h, hs.cleared, 0) != cudaSuccess) return drain(gemm::kErrLaunch);
  for (int64_t i = 0; i < tr; ++i) {
    int64_t b0, b1;
    group_rows(i, b0, b1);
    const int64_t r0 = b0 * rows, n = (b1 * rows < M ? b1 * rows : M) - r0;
    const unsigned target = gemm::tc_stream_done_target(N, b1 - b0);
    if (target >= gemm::kStreamRelease) return drain(gemm::kErrInvalidArg);  // never: < 2^27
    if (ops.wait(hs.d2h, dptr(c_done + i), target, CU_STREAM_WAIT_VALUE_GEQ) != CUDA_SUCCESS)
      return drain(gemm::kErrLaunch);
    if (cudaMemcpy2DAsync(host.C + r0 * host.ldc, host.ldc * 4, dC + r0 * dldc, dldc * 4, N * 4, n,
                          cudaMemcpyDeviceToHost, hs.d2h) != cudaSuccess)
      return drain(gemm::kErrLaunch);
  }
  // Bounded wait for the last copy of C. The kernel raises every counter
  // when it gives up, so the return stream always gets through; should it
  // not, after twice the kernel's own limit the counters are raised from the
  // copy stream (which waits on nothing) and the call reports a timeout.
  const auto t0 = std::chrono::steady_clock::now();
  const double kernel_limit_s =
      timeout_ns > 0 ? 1e-9 * static_cast<double>(timeout_ns) : 2.0 + 2e-6 * static_cast<double>(K);
  const double limit_s = 2.0 * kernel_limit_s + 1.0;
  for (;;) {
    const cudaError_t q = cudaStreamQuery(hs.d2h);
    if (q == cudaSuccess) break;
    if (q != cudaErrorNotReady) return drain(gemm::kErrLaunch);
    if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > limit_s) {
      for (int64_t r = 0; r < tr; ++r)
        ops.write(hs.h2d, dptr(c_done + r), gemm::kStreamRelease, CU_STREAM_WRITE_VALUE_DEFAULT);
      drain(0);
      const int tst = gemm::tc_poll_status(hs.stream);
      return tst != gemm::kOk ? tst : gemm::kErrTimeout;
    }
    std::this_thread::yield();
  }
  return gemm::tc_poll_status(hs.stream);
}

// Checked build: the index-check records of every kernel translation unit
// (read after the caller synchronised). Returns the total count of recorded
// violations (-1 if a record could not be read), *first the first record of
// the first unit that has one; clear: reset the records.
long long take_index_faults(bool clear, gemm::IndexFault *first) {
  if (!GEMM_F32_INDEX_CHECKS) {
    if (first != nullptr) *first = gemm::IndexFault{0u, 0, 0, 0};
    return 0;
  }
  int (*const takers[])(gemm::IndexFault *, bool) = {
      gemm::tc_index_fault_take, gemm::simt_index_fault_take, gemm::pack_index_fault_take,
      gemm::transpose_index_fault_take, gemm::reduce_index_fault_take};
  long long total = 0;
  bool have = false;
  for (auto take : takers) {
    gemm::IndexFault f = {0u, 0, 0, 0};
    if (take(&f, clear) != gemm::kOk) return -1;
    total += f.count;
    if (f.count > 0 && !have) {
      have = true;
      if (first != nullptr) *first = f;
    }
  }
  if (!have && first != nullptr) *first = gemm::IndexFault{0u, 0, 0, 0};
  return total;
}

}  // namespace

extern "C" {

int gemm_f32_ex(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                int64_t ldb, float *C, int64_t ldc, int mode, int kernel, void *stream) {
  const GemmArgs a{M, N, K, A, lda, B, ldb, C, ldc};
  return run(a, mode, kernel, static_cast<cudaStream_t>(stream));
}

int gemm_f32_general(int order, int transa, int transb, int64_t M, int64_t N, int64_t K,
                     float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                     float beta, float *C, int64_t ldc, int mode, int kernel, void *stream) {
  GemmArgs a{M, N, K, A, lda, B, ldb, C, ldc};
  if (order == GEMM_ROW_MAJOR) {
    a.opa = transa;
    a.opb = transb;
  } else if (order == GEMM_COL_MAJOR) {
    // A column-major matrix is the row-major storage of its transpose, so
    // C = op(A) op(B) in column-major order is C^T = op(B)^T op(A)^T in
    // row-major order: swap the operands and their flags and exchange M, N.
    a = GemmArgs{N, M, K, B, ldb, A, lda, C, ldc};
    a.opa = transb;
    a.opb = transa;
  } else {
    return GEMM_ERR_INVALID_ARG;
  }
  a.alpha = alpha;
  a.beta = beta;
  return run(a, mode, kernel, static_cast<cudaStream_t>(stream));
}

int gemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
             int64_t ldb, float *C, int64_t ldc, int mode, void *stream) {
  return gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, mode, GEMM_KERNEL_AUTO, stream);
}

int gemm_f32_select(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                    int64_t ldb, float *C, int64_t ldc, int mode, int kernel) {
  const GemmArgs a{M, N, K, A, lda, B, ldb, C, ldc};
  bool noop = false;
  const int st = validate(a, mode, &noop);
  if (st != gemm::kOk) return -st;
  return select_kernel(a, mode, kernel);
}

// gemm_f32_host, and its failure self-test (skip_block, timeout_ns: see
// host_streamed). Internal: not exported.
static int gemm_f32_host_impl(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                              const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                              int64_t skip_block, unsigned long long timeout_ns);

int gemm_f32_host(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                  int64_t ldb, float *C, int64_t ldc, int mode) {
  return gemm_f32_host_impl(M, N, K, A, lda, B, ldb, C, ldc, mode, -1, 0);
}

int gemm_f32_selftest_host_missing_block(int64_t M, int64_t N, int64_t K, const float *A,
                                         int64_t lda, const float *B, int64_t ldb, float *C,
                                         int64_t ldc, int64_t timeout_ns) {
  if (timeout_ns < 1000000 || timeout_ns > 10000000000LL || K < 16) return GEMM_ERR_INVALID_ARG;
  if (stream_value_ops().write == nullptr) return GEMM_ERR_INVALID_ARG;
  // The last block of A: the kernel's waits for it run out.
  const int64_t tiles_m = (M + gemm::kStreamRows - 1) / gemm::kStreamRows;
  int64_t per_copy = (tiles_m + 3) / 4;
  per_copy = per_copy > 4 ? 4 : (per_copy < 1 ? 1 : per_copy);
  const int64_t last = (tiles_m + per_copy - 1) / per_copy - 1;
  return gemm_f32_host_impl(M, N, K, A, lda, B, ldb, C, ldc, GEMM_F32_EXACT, last,
                            static_cast<unsigned long long>(timeout_ns));
}

static int gemm_f32_host_impl(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                              const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                              int64_t skip_block, unsigned long long timeout_ns) {
  const GemmArgs host{M, N, K, A, lda, B, ldb, C, ldc};
  bool noop = false;
  int st = validate(host, mode, &noop);
  if (st != gemm::kOk || noop) return st;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;

  HostState &hs = g_host[dev];
  std::lock_guard<std::mutex> g(hs.mu);
  st = host_state_init(hs);
  if (st != gemm::kOk) return st;

  // Device layout: pitches padded to multiples of 4 elements (16 bytes), each
  // matrix starting on a 256-byte boundary.
  const int64_t dlda = round_up4(K > 0 ? K : 1), dldb = round_up4(N), dldc = round_up4(N);
  auto up256 = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t bytes_a = up256(static_cast<size_t>(M * dlda) * 4);
  const size_t bytes_b = up256(static_cast<size_t>((K > 0 ? K : 1) * dldb) * 4);
  const size_t bytes_c = up256(static_cast<size_t>(M * dldc) * 4);
  const size_t need = bytes_a + bytes_b + bytes_c;
  if (need > hs.cap_bytes) {
    if (hs.buf) cudaFree(hs.buf);
    hs.buf = nullptr;
    hs.cap_bytes = 0;
    if (cudaMalloc(&hs.buf, need) != cudaSuccess) return gemm::kErrLaunch;
    hs.cap_bytes = need;
  }
  uint8_t *base = reinterpret_cast<uint8_t *>(hs.buf);
  float *dA = reinterpret_cast<float *>(base);
  float *dB = reinterpret_cast<float *>(base + bytes_a);
  float *dC = reinterpret_cast<float *>(base + bytes_a + bytes_b);

  // Exact mode from K = 16 (where gemm_f32 runs the 3xTF32 kernel) takes one
  // launch fed while it runs, when the driver offers stream memory
  // operations: 0.96 against 1.02 ms at 4096^3, where the row chunks' GEMMs
  // (127.5 us each, against 97.5 for a quarter of one launch) set the pace.
  // One TF32 pass, bound by the host link either way, keeps the row chunks
  // (0.90 against 0.92 ms), as do the FP32 SIMT mode, K == 0 and exact mode
  // below K = 16.
  if (mode == GEMM_F32_EXACT && K >= 16 && stream_value_ops().write != nullptr)
    return host_streamed(hs, host, sms, dA, dlda, dB, dldb, dC, dldc, skip_block, timeout_ns);

  // Row chunks pipelined over three streams: B, then A chunk by chunk, go
  // host to device on one; each chunk's GEMM starts on the compute stream as
  // soon as its rows of A (and all of B) have landed; its rows of C go back
  // on the third, so the copies of later and earlier chunks overlap the
  // GEMM of this one. Chunks are a quarter of M in whole 256-row tiles and
  // at least 1024 rows: a row chunk is a smaller GEMM that keeps fewer SMs
  // busy (4096^3 as 8 chunks of 512 rows takes 1.5x the time of one call,
  // as 4 of 1024 rows 1.2x). Every chunk needs all of B, so B goes first, in
  // two halves of whole rows around the first chunk of A (when K >= 512):
  // the first chunk's GEMM runs over the first half of K while the second
  // half of B is still on its way, then adds the second half (beta = 1), so
  // that only half of that GEMM waits behind the whole of B.
  int64_t chunk = (M + 3) / 4;
  chunk = (chunk + 255) / 256 * 256;
  if (chunk < 1024) chunk = 1024;
  if ((M + chunk - 1) / chunk > kHostMaxChunks) chunk = (M + kHostMaxChunks - 1) / kHostMaxChunks;
  const int nchunks = static_cast<int>((M + chunk - 1) / chunk);
  // First half of B: rows [0, k1), a multiple of 32 (whole k-blocks, and a
  // 16-byte aligned offset into the rows of A); 0 when K is too short.
  const int64_t k1 = K >= 512 ? (K / 2) / 32 * 32 : 0;
  // On an error once copies are queued, wait for all queued work before
  // returning, so that no copy reads or writes the caller's buffers after
  // the call has returned.
  auto drain = [&hs](int code) {
    cudaStreamSynchronize(hs.h2d);
    cudaStreamSynchronize(hs.stream);
    cudaStreamSynchronize(hs.d2h);
    return code;
  };
  auto copy_b_rows = [&](int64_t r0, int64_t rows) {
    return cudaMemcpy2DAsync(dB + r0 * dldb, dldb * 4, B + r0 * ldb, ldb * 4, N * 4, rows,
                             cudaMemcpyHostToDevice, hs.h2d);
  };
  if (K > 0 && copy_b_rows(0, k1 > 0 ? k1 : K) != cudaSuccess) return drain(gemm::kErrLaunch);
  for (int c = 0; c < nchunks; ++c) {
    const int64_t r0 = c * chunk, rows = (M - r0 < chunk) ? M - r0 : chunk;
    if (K > 0 && cudaMemcpy2DAsync(dA + r0 * dlda, dlda * 4, A + r0 * lda, lda * 4, K * 4, rows,
                                   cudaMemcpyHostToDevice, hs.h2d) != cudaSuccess)
      return drain(gemm::kErrLaunch);
    if (cudaEventRecord(hs.a_in[c], hs.h2d) != cudaSuccess ||
        cudaStreamWaitEvent(hs.stream, hs.a_in[c], 0) != cudaSuccess)
      return drain(gemm::kErrLaunch);
    if (c == 0 && k1 > 0) {
      // The second half of B follows the first chunk of A.
      if (copy_b_rows(k1, K - k1) != cudaSuccess || cudaEventRecord(hs.b_hi, hs.h2d) != cudaSuccess)
        return drain(gemm::kErrLaunch);
      GemmArgs lo{rows, N, k1, dA, dlda, dB, dldb, dC, dldc};
      st = run(lo, mode, GEMM_KERNEL_AUTO, hs.stream);
      if (st != gemm::kOk) return drain(st);
      if (cudaStreamWaitEvent(hs.stream, hs.b_hi, 0) != cudaSuccess) return drain(gemm::kErrLaunch);
      GemmArgs hi{rows, N, K - k1, dA + k1, dlda, dB + k1 * dldb, dldb, dC, dldc};
      hi.beta = 1.0f;
      st = run(hi, mode, GEMM_KERNEL_AUTO, hs.stream);
    } else {
      const GemmArgs d{rows, N, K, dA + r0 * dlda, dlda, dB, dldb, dC + r0 * dldc, dldc};
      st = run(d, mode, GEMM_KERNEL_AUTO, hs.stream);
    }
    if (st != gemm::kOk) return drain(st);
    if (cudaEventRecord(hs.c_done[c], hs.stream) != cudaSuccess ||
        cudaStreamWaitEvent(hs.d2h, hs.c_done[c], 0) != cudaSuccess ||
        cudaMemcpy2DAsync(C + r0 * ldc, ldc * 4, dC + r0 * dldc, dldc * 4, N * 4, rows,
                          cudaMemcpyDeviceToHost, hs.d2h) != cudaSuccess)
      return drain(gemm::kErrLaunch);
  }
  if (cudaStreamSynchronize(hs.d2h) != cudaSuccess) return gemm::kErrLaunch;
  return gemm::tc_poll_status(hs.stream);
}

int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb, float *C, int64_t ldc, int mode, void *stream) {
  const GemmArgs a{M, N, K, A, lda, B, ldb, C, ldc};
  bool noop = false;
  int st = validate(a, mode, &noop);
  if (st != gemm::kOk || noop) return st;
  const int k = select_kernel(a, mode, GEMM_KERNEL_AUTO, /*can_pack=*/false);
  if (k < 0) return -k;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.K == 0) {
    if (cudaMemset2DAsync(a.C, static_cast<size_t>(a.ldc) * 4, 0, static_cast<size_t>(a.N) * 4,
                          static_cast<size_t>(a.M), s) != cudaSuccess)
      return gemm::kErrLaunch;
    return gemm::kOk;
  }
  if (k == GEMM_KERNEL_SIMT) return gemm::simt_launch(a, sms, false, s);  // no workspace
  return gemm::tc_launch_noalloc(a, mode == GEMM_F32_EXACT, k == GEMM_KERNEL_TC_LSU, sms, s);
}

int reduce_f32_sum(int64_t n, const float *x, float *out, int groups, void *stream) {
  if (n < 0 || n > (int64_t{1} << 40) || groups < 0 || groups > 65535) return GEMM_ERR_INVALID_ARG;
  if (out == nullptr || reinterpret_cast<uintptr_t>(out) % 4 != 0) return GEMM_ERR_INVALID_ARG;
  if (n > 0) {
    if (x == nullptr || reinterpret_cast<uintptr_t>(x) % 4 != 0) return GEMM_ERR_INVALID_ARG;
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), x1 = x0 + static_cast<uintptr_t>(n) * 4;
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out);
    if (ranges_overlap(o0, o0 + 4, x0, x1)) return GEMM_ERR_ALIAS;
  }
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n == 0) return gemm::reduce_launch(0, x, out, 1, nullptr, s);
  const int g = groups > 0 ? groups : gemm::reduce_default_groups(sms);
  void *partials = nullptr;
  st = gemm::pool_alloc(&partials, static_cast<size_t>(g) * sizeof(float), s);
  if (st != gemm::kOk) return st;
  st = gemm::reduce_launch(n, x, out, g, static_cast<float *>(partials), s);
  const int fst = gemm::pool_free(partials, s);
  return st != gemm::kOk ? st : fst;
}

const char *gemm_f32_status_string(int status) {
  switch (status) {
    case GEMM_OK:
      return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG:
      return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED_DEVICE:
      return "GEMM_ERR_UNSUPPORTED_DEVICE";
    case GEMM_ERR_LAUNCH:
      return "GEMM_ERR_LAUNCH";
    case GEMM_ERR_TIMEOUT:
      return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_ALIAS:
      return "GEMM_ERR_ALIAS";
    case GEMM_ERR_INDEX:
      return "GEMM_ERR_INDEX";
    default:
      return "GEMM_ERR_UNKNOWN";
  }
}

int gemm_f32_measure_peaks(double *tf32_tflops, double *fp32_tflops, double *tf32_sm_mhz,
                           double *fp32_sm_mhz) {
  if (tf32_tflops == nullptr || fp32_tflops == nullptr || tf32_sm_mhz == nullptr ||
      fp32_sm_mhz == nullptr)
    return GEMM_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  const int st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return GEMM_ERR_LAUNCH;
  const int r = gemm::probe_peaks(sms, tf32_tflops, fp32_tflops, tf32_sm_mhz, fp32_sm_mhz, s);
  cudaStreamDestroy(s);
  return r;
}

int gemm_f32_poll_device_status(void *stream) {
  int dev = 0, sms = 0;
  const int st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  const int tst = gemm::tc_poll_status(static_cast<cudaStream_t>(stream));
  if (tst != gemm::kOk || !GEMM_F32_INDEX_CHECKS) return tst;
  // Checked build: a recorded index violation, left for take_index_fault.
  if (take_index_faults(false, nullptr) > 0) return GEMM_ERR_INDEX;
  return gemm::kOk;
}

int gemm_f32_checked_build(void) { return GEMM_F32_INDEX_CHECKS ? 1 : 0; }

int gemm_f32_take_index_fault(void *stream, long long *count, int *site, long long *offset,
                              long long *extent) {
  if (count == nullptr || site == nullptr || offset == nullptr || extent == nullptr)
    return GEMM_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  const int st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GEMM_ERR_LAUNCH;
  gemm::IndexFault first = {0u, 0, 0, 0};
  const long long n = take_index_faults(true, &first);
  if (n < 0) return GEMM_ERR_LAUNCH;
  *count = n;
  *site = first.site;
  *offset = first.offset;
  *extent = first.extent;
  return GEMM_OK;
}

const char *gemm_f32_index_site_name(int site) {
  switch (site) {
    case gemm::kSiteNone:
      return "none";
    case gemm::kSiteCStore:
      return "C store";
    case gemm::kSitePartialWrite:
      return "partial slot write";
    case gemm::kSitePartialRead:
      return "partial slot read";
    case gemm::kSiteCounter:
      return "split-tile counter";
    case gemm::kSiteBand:
      return "cluster-split band (shared memory)";
    case gemm::kSiteLoadA:
      return "A load";
    case gemm::kSiteLoadB:
      return "B load";
    case gemm::kSiteCopySrc:
      return "operand copy source";
    case gemm::kSiteCopyDst:
      return "operand copy destination";
    case gemm::kSiteReduceIn:
      return "reduction input";
    case gemm::kSiteReducePartial:
      return "reduction partial";
    case gemm::kSiteReduceOut:
      return "reduction output";
    default:
      return "unknown";
  }
}

int gemm_f32_selftest_index_check(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                  const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                                  int kernel, void *stream) {
  if (!GEMM_F32_INDEX_CHECKS) return GEMM_ERR_INVALID_ARG;  // nothing to check in this build
  GemmArgs a{M, N, K, A, lda, B, ldb, C, ldc};
  bool noop = false;
  int st = validate(a, mode, &noop);
  if (st != gemm::kOk) return st;
  if (noop || M < 2 || K < 1) return GEMM_ERR_INVALID_ARG;
  // C declared one row short: every access to its last row fails the check.
  a.c_extent = gemm::matrix_extent(M - 1, N, ldc);
  return run(a, mode, kernel, static_cast<cudaStream_t>(stream));
}

int gemm_f32_selftest_wait_timeout(int64_t timeout_ns, void *stream) {
  if (timeout_ns < 1000000 || timeout_ns > 10000000000LL) return GEMM_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  const int st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  return gemm::tc_selftest_wait_timeout(timeout_ns, static_cast<cudaStream_t>(stream));
}

int gemm_f32_selftest_stalled_gemm(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                   const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                                   int64_t timeout_ns, void *stream) {
  if (timeout_ns < 1000000 || timeout_ns > 10000000000LL) return GEMM_ERR_INVALID_ARG;
  if (mode != GEMM_F32_EXACT && mode != GEMM_F32_TF32) return GEMM_ERR_INVALID_ARG;
  const GemmArgs a{M, N, K, A, lda, B, ldb, C, ldc};
  bool noop = false;
  int st = validate(a, mode, &noop);
  if (st != gemm::kOk) return st;
  if (noop) return GEMM_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != gemm::kOk) return st;
  return gemm::tc_selftest_stalled_gemm(a, mode == GEMM_F32_EXACT, timeout_ns, sms,
                                        static_cast<cudaStream_t>(stream));
}

}  // extern "C"
