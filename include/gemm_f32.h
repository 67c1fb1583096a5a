/*
 * gemm_f32.h -- C ABI of libgemm_f32.so: dense row-major single-precision
 * matrix multiplication C = A x B on an NVIDIA GB300 (sm_103a).
 *
 * Operation. A is M x K, B is K x N, C is M x N, all fp32 and row-major with
 * leading dimensions lda, ldb, ldc counted in elements (element (i, j) of A is
 * A[i * lda + j]). Every call overwrites C with the product:
 *
 *     C[i][j] = sum_{k < K} A[i][k] * B[k][j]
 *
 * This is the product that "Optimizing a WebGPU Matmul Kernel using
 * Subgroups" builds up one output cell at a time (section 1, "Naive"; its
 * later sections tile, vectorise and hand it to matrix units), with the
 * M x K by K x N problem statement of "WebGPU WGSL Compute Shaders: Custom
 * Matrix Multiplication (GEMM) Optimization Guide" (section 1) and the caller
 * owned A, B (read) and C (written) buffers of its section 5 dispatch routine.
 * C is overwritten, never accumulated into, as in every kernel on those pages.
 * Out-of-range tile elements contribute zero and are never stored, the
 * zero-filled boundary of section 4 of the same guide.
 *
 * Accuracy classes (stated per element against the exact product, with
 * S = |A| x |B|):
 *   GEMM_F32_EXACT       |C - AB| <= 2 K 2^-24 S  (FP32 class). Tensor cores
 *                        with a 3xTF32 split (hi/lo operand decomposition),
 *                        or the SIMT FP32 kernel when K < 16.
 *   GEMM_F32_TF32        |C - AB| <= 2 K 2^-11 S  (TF32 class). One TF32 pass
 *                        on the tensor cores; the low 13 mantissa bits of each
 *                        operand are dropped by the hardware.
 *   GEMM_F32_EXACT_SIMT  FP32 class, always on the SIMT FP32 kernel.
 * No call returns a result of a lower class than the mode asks for.
 *
 * Streams and ownership. All matrix pointers passed to gemm_f32 and
 * gemm_f32_ex are DEVICE pointers owned by the caller; the library keeps no
 * reference to them after the call returns. `stream` is a cudaStream_t passed
 * as void* (NULL = the legacy default stream). The call is stream ordered: it
 * enqueues work and returns without synchronising. When the schedule splits
 * the k range of some output tiles between SMs (stream-K), the call takes a
 * workspace of at most two 128 KiB partial tiles per SM from a stream-ordered
 * memory pool that the library creates on each device and never shrinks, and
 * returns it to the pool behind the kernel on the same stream; calls on
 * different streams therefore never share it. gemm_f32_noalloc avoids even
 * that.
 *
 * Errors are returned synchronously as gemm_f32_status codes. Argument errors
 * are detected on the host before anything is enqueued, and no CUDA call is
 * made for them. A kernel whose pipeline wait runs out of time (a hardware or
 * scheduling failure; never expected) records GEMM_ERR_TIMEOUT in a device
 * status word, leaves C unspecified and exits cleanly; read it with
 * gemm_f32_poll_device_status.
 *
 * Thread safety: all entry points may be called from several host threads.
 */
#ifndef GEMM_F32_H
#define GEMM_F32_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_F32_EXACT = 0,      /* FP32-accurate: 3xTF32 tensor cores (SIMT if K < 16) */
    GEMM_F32_TF32 = 1,       /* single-pass TF32 on tensor cores */
    GEMM_F32_EXACT_SIMT = 2  /* FP32-accurate on the SIMT FP32 kernel */
} gemm_f32_mode;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,         /* bad size, leading dimension, pointer, mode or kernel */
    GEMM_ERR_UNSUPPORTED_DEVICE = 2,  /* current device is not compute capability 10.3 */
    GEMM_ERR_LAUNCH = 3,              /* a CUDA launch or API call failed */
    GEMM_ERR_TIMEOUT = 4,             /* a device-side pipeline wait ran out of time */
    GEMM_ERR_ALIAS = 5,               /* C overlaps A or B */
    GEMM_ERR_INDEX = 6                /* checked build: a device-side index check failed */
} gemm_f32_status;

/* Kernel choice for gemm_f32_ex. */
typedef enum {
    GEMM_KERNEL_AUTO = 0,    /* what gemm_f32 picks */
    GEMM_KERNEL_SIMT = 1,    /* SIMT FP32 register-tiled kernel (exact modes only) */
    GEMM_KERNEL_TC_TMA = 2,  /* tcgen05 kernel fed by TMA (operands copied first if TMA
                                cannot read them as given; see gemm_f32_ex) */
    GEMM_KERNEL_TC_LSU = 3   /* tcgen05 kernel fed by plain loads (any strides) */
} gemm_f32_kernel;

/*
 * gemm_f32 -- C = A x B, stream ordered.
 *   M, N, K   sizes, >= 0. M == 0 or N == 0 is a no-op; K == 0 sets C to zero
 *             (the empty sum).
 *   A, lda    device pointer to M x K fp32, 4-byte aligned, lda >= max(1, K)
 *   B, ldb    device pointer to K x N fp32, 4-byte aligned, ldb >= max(1, N)
 *   C, ldc    device pointer to M x N fp32, 4-byte aligned, ldc >= max(1, N);
 *             must not overlap A or B (GEMM_ERR_ALIAS)
 *   mode      a gemm_f32_mode
 *   stream    cudaStream_t as void*
 * Sizes and leading dimensions must stay below 2^31 elements, and the span
 * of each matrix, (rows - 1) x ld + cols elements, at most 2^44.
 * Returns a gemm_f32_status. Stream-ordered and non-blocking.
 */
int gemm_f32(int64_t M, int64_t N, int64_t K,
             const float *A, int64_t lda,
             const float *B, int64_t ldb,
             float *C, int64_t ldc,
             int mode, void *stream);

/*
 * gemm_f32_ex -- gemm_f32 with an explicit kernel choice (a gemm_f32_kernel).
 * GEMM_KERNEL_AUTO behaves exactly like gemm_f32. A kernel that cannot serve
 * the arguments returns GEMM_ERR_INVALID_ARG: GEMM_KERNEL_SIMT with mode
 * GEMM_F32_TF32 (it would change the accuracy class). TMA reads operands
 * whose base is 16-byte aligned and whose leading dimension is a multiple of
 * 4; GEMM_KERNEL_TC_TMA (and AUTO, for the tensor-core modes) copies any
 * other operand first into a workspace with that layout, taken from the
 * library's stream-ordered pool on `stream` (rows x round_up(cols, 4) floats
 * per copied operand) and returned behind the GEMM: one read and one write of
 * the operand in HBM. GEMM_KERNEL_TC_LSU reads any layout in place with plain
 * loads instead (slower per flop, no copy). Mode GEMM_F32_EXACT with a
 * tensor-core kernel forced runs 3xTF32 for every K, including K < 16.
 */
int gemm_f32_ex(int64_t M, int64_t N, int64_t K,
                const float *A, int64_t lda,
                const float *B, int64_t ldb,
                float *C, int64_t ldc,
                int mode, int kernel, void *stream);

/* Storage order and operand transposition for gemm_f32_general. */
typedef enum {
    GEMM_ROW_MAJOR = 0,  /* element (i, j) of a matrix with pitch ld at [i * ld + j] */
    GEMM_COL_MAJOR = 1   /* element (i, j) at [j * ld + i] (BLAS / LAPACK storage) */
} gemm_f32_order;

typedef enum {
    GEMM_OP_N = 0,  /* op(X) = X */
    GEMM_OP_T = 1   /* op(X) = X^T: the operand is supplied transposed */
} gemm_f32_op;

/*
 * gemm_f32_general -- C = alpha * op(A) op(B) + beta * C, stream ordered.
 *
 * The general form of gemm_f32: op(A) is M x K, op(B) is K x N, C is M x N.
 * Transposed operands are the layouts of "Optimizing a WebGPU Matmul Kernel
 * using Subgroups", section 7 (B supplied transposed, N x K, so that both
 * operands are read along k) and of the column-major (BLAS) storage that
 * "WebGPU 计算着色器矩阵乘法优化：从 Naive 到 Tiled 深度实战" ("工程实践建议")
 * advises adapting the indexing to. alpha and beta are not on the pages,
 * whose kernels overwrite C; they are the usual scale of the product and of
 * the previous C.
 *   order     a gemm_f32_order; it applies to A, B and C alike.
 *   transa    a gemm_f32_op. Stored A: M x K for GEMM_OP_N, K x M for
 *             GEMM_OP_T, with lda >= max(1, columns of the stored A in
 *             row-major order / rows in column-major order).
 *   transb    a gemm_f32_op. Stored B: K x N for GEMM_OP_N, N x K for
 *             GEMM_OP_T, with ldb likewise.
 *   alpha     scale of the product. alpha == 0 or K == 0: A and B are not
 *             read and C = beta * C.
 *   beta      scale of the previous C. beta == 0: C is not read, so its
 *             previous contents (NaN included) do not matter.
 *   C, ldc    ldc >= max(1, N) (row-major) or max(1, M) (column-major).
 *   mode, kernel, stream   as for gemm_f32_ex.
 * A column-major call is the row-major call on the transposes (C^T =
 * op(B)^T op(A)^T): the library swaps the operands and their flags. When a
 * row-major call has transa == GEMM_OP_T (column-major: transb ==
 * GEMM_OP_T), the TMA-fed tensor-core kernel (GEMM_KERNEL_TC_TMA, which AUTO
 * picks) runs on a row-major copy of op(A) that a transpose kernel writes
 * first, like any operand TMA cannot read as given (see gemm_f32_ex);
 * GEMM_KERNEL_TC_LSU instead transposes each tile of A as it stages it,
 * with no workspace. Accuracy
 * classes apply to alpha * op(A) op(B) with S = |op(A)| |op(B)| scaled by
 * |alpha|, plus one rounding of the scale-and-add.
 * gemm_f32(...) is gemm_f32_general(GEMM_ROW_MAJOR, GEMM_OP_N, GEMM_OP_N,
 * M, N, K, 1, A, lda, B, ldb, 0, C, ldc, mode, GEMM_KERNEL_AUTO, stream).
 * Returns a gemm_f32_status; errors as for gemm_f32 (an unknown order or op
 * is GEMM_ERR_INVALID_ARG).
 */
int gemm_f32_general(int order, int transa, int transb,
                     int64_t M, int64_t N, int64_t K,
                     float alpha,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float beta,
                     float *C, int64_t ldc,
                     int mode, int kernel, void *stream);

/*
 * gemm_f32_select -- the kernel gemm_f32_ex would run for these arguments (a
 * gemm_f32_kernel value, never AUTO), or a negative gemm_f32_status if the
 * arguments are invalid. Host-only: it inspects sizes, leading dimensions and
 * pointer alignment and makes no CUDA call.
 */
int gemm_f32_select(int64_t M, int64_t N, int64_t K,
                    const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float *C, int64_t ldc,
                    int mode, int kernel);

/*
 * gemm_f32_host -- C = A x B for matrices in HOST memory (pageable or pinned).
 * Copies A and B to device buffers that the library owns and reuses (grown on
 * demand, one set per device, held until process exit), computes on
 * library-owned streams of the current device, copies C back and waits for
 * completion. Blocking. Copies and compute overlap (page-locked host memory
 * copies fastest); when K >= 512, B goes in two halves of whole rows, the
 * second after the first rows of A, so that the first GEMM work runs over
 * the first half of K while the second half is on its way.
 *   GEMM_F32_EXACT with K >= 16 (the 3xTF32 kernel): one launch of the
 *     kernel over all of C, started before any operand has landed. A goes
 *     to the device in blocks of up to 1024 rows; after each block (and each
 *     half of B) the copy stream writes a word in device memory, for which
 *     the kernel waits (bounded, as its pipeline waits are) before it reads
 *     those rows. The kernel counts the stored tiles of each block of C, and
 *     the return stream copies a block to the host as soon as its count is
 *     complete. Needs the driver's stream memory operations; without them,
 *     the row chunks below.
 *   Other modes and sizes: row chunks (a quarter of M, at least 1024 rows):
 *     B and then each chunk of A go to the device on one stream, each
 *     chunk's GEMM (a gemm_f32 call) starts when its rows have landed, and
 *     its rows of C come back on another stream while later chunks compute;
 *     with the two halves of B, the first chunk's GEMM adds the second half
 *     of K (beta = 1) once it has landed.
 * Results meet the accuracy class of the mode; they may differ in the last
 * bits from one gemm_f32 call on the whole matrices, whose split of the work
 * differs. A kernel that gives up (GEMM_ERR_TIMEOUT) releases the copies of
 * C, so the call returns; a wait by the host for them is bounded too. Same size, leading-dimension, mode and alias rules as gemm_f32
 * (alias checked on the host ranges). Device-side leading dimensions are
 * padded to multiples of 4 so the TMA-fed kernels apply at any K and N.
 * Calls on one device are serialised by a lock. On every return, success
 * or error, no copy the call queued still reads or writes the host buffers.
 */
int gemm_f32_host(int64_t M, int64_t N, int64_t K,
                  const float *A, int64_t lda,
                  const float *B, int64_t ldb,
                  float *C, int64_t ldc,
                  int mode);

/* Bytes of the fixed device array that gemm_f32_noalloc works in (40 MiB). */
#define GEMM_F32_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)

/*
 * gemm_f32_noalloc -- gemm_f32 without any device memory allocation. (The
 * pages have no counterpart: their kernels need no scratch memory.)
 *
 * For callers that must not allocate device memory while they run: programs
 * that hand nearly all device memory to their own allocator at start-up (so
 * a pool allocation on the caller's stream could fail), and latency- or
 * budget-critical loops that must keep the process's device footprint and
 * allocator state fixed once set up. gemm_f32 takes its stream-K workspace
 * (partial sums of output tiles whose k range is shared between SMs) from
 * the library's stream-ordered memory pool; this entry point runs the same
 * kernels and schedule but keeps that workspace in a fixed array of
 * GEMM_F32_NOALLOC_SCRATCH_BYTES that is part of the library's device image:
 * every GPU that loads the library holds it until the process exits.
 *
 * Arguments, modes, layout and errors are those of gemm_f32 (device
 * pointers owned by the caller, stream ordered, non-blocking), and results
 * are the same. It never copies operands into a workspace: those TMA
 * cannot read as given (see gemm_f32_ex) go to the tensor-core kernel fed by
 * plain loads. In addition it returns GEMM_ERR_INVALID_ARG, before
 * enqueuing anything, for a problem whose workspace would not fit in the
 * array. The workspace holds at most two 128 KiB partial tiles per SM plus a
 * few counters (under 39 MiB on a 152-SM GB300, whatever the shape), so on
 * such a device every valid problem fits; the check guards larger devices.
 *
 * Set-up. The array belongs to the library's tensor-core code module, which
 * the CUDA runtime places in device memory when it first needs it on a
 * device: with CUDA's lazy module loading (the default) that is the first
 * tensor-core call of any entry point, or the first gemm_f32_noalloc call,
 * whose set-up also looks up the array's device address (with that device
 * current). So make one gemm_f32_noalloc call on each device before handing
 * device memory to another allocator and before any stream capture, or set
 * CUDA_MODULE_LOADING=EAGER so that the array is placed when the context is
 * created. The address is kept for the life of the process: calls after
 * cudaDeviceReset on that device are not supported.
 *
 * Every call on a device uses the same array and leaves its contents behind;
 * the call itself clears what must start at zero. Calls whose work overlaps
 * on the GPU (different streams, or different host threads) race on the
 * array and give wrong results: serialise them.
 */
int gemm_f32_noalloc(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float *C, int64_t ldc,
                     int mode, void *stream);

/*
 * gemm_f32_measure_peaks -- measurement helper, not part of any computation:
 * runs an MMA-only kernel (tcgen05.mma kind::tf32, 128 x 256 x 8, operands
 * resident in shared memory and filled with non-zero values, one CTA per SM)
 * and an FFMA-only kernel (independent fused multiply-add chains, 1024
 * threads per SM) on the current device and returns, through the four
 * pointers (host memory), the rates they reach in TFLOP/s and the median SM
 * clock in MHz each kernel's CTAs ran at (SM clock ticks over wall time,
 * measured inside the kernel), so that a rate can be compared with another
 * measured at a different clock. Blocking; takes a fraction of a second. The
 * pages have no counterpart: they time their kernels against no peak.
 */
int gemm_f32_measure_peaks(double *tf32_tflops, double *fp32_tflops,
                           double *tf32_sm_mhz, double *fp32_sm_mhz);

/* gemm_f32_status_string -- static, NUL-terminated name of a status code. */
const char *gemm_f32_status_string(int status);

/*
 * gemm_f32_poll_device_status -- synchronise `stream`, then return and clear
 * the device status word of the current device (GEMM_OK if no kernel has
 * recorded an error since the last poll). Returns GEMM_ERR_LAUNCH if the
 * synchronisation itself fails. In the checked build (below) it returns
 * GEMM_ERR_INDEX when no wait has timed out but an index check has failed
 * since the last gemm_f32_take_index_fault; the record stays for that call.
 */
int gemm_f32_poll_device_status(void *stream);

/*
 * The checked build. libgemm_f32_checked.so exports the same functions as
 * libgemm_f32.so, compiled with device-side index checks: before every
 * global-memory access that a kernel addresses with its own index
 * arithmetic -- plain loads of A and B, stores and beta reads of C, the
 * partial-sum slots and counters of split tiles, the operand copies, the
 * reduction -- it compares the element offset with the extent the call
 * declared for that buffer ((rows - 1) x pitch + columns for a matrix, the
 * allocation for a library workspace). A failed check skips the access (no
 * fault, no trap; the kernel carries on) and counts it; the first one of
 * each kernel source file is recorded. TMA copies are bounded by their
 * tensor maps in hardware and need no check. The checks cost time; the
 * regular library has none (index checks compile to nothing).
 *
 * gemm_f32_checked_build -- 1 in the checked build, 0 in the regular one.
 */
int gemm_f32_checked_build(void);

/*
 * gemm_f32_take_index_fault -- synchronise `stream`, then read and reset the
 * index-check records of the current device: *count = failed checks since
 * the last call, and the first recorded one's *site (a GEMM_F32 site code,
 * see gemm_f32_index_site_name), element *offset and declared *extent (all
 * 0 when *count is 0). Always *count = 0 in the regular build. Returns
 * GEMM_OK, GEMM_ERR_INVALID_ARG for a null output pointer, GEMM_ERR_LAUNCH
 * if the synchronisation or a read fails. Outputs are host pointers.
 */
int gemm_f32_take_index_fault(void *stream, long long *count, int *site, long long *offset,
                              long long *extent);

/* gemm_f32_index_site_name -- static, NUL-terminated name of an index-check
 * site code (1 C store, 2 partial slot write, 3 partial slot read, 4
 * split-tile counter, 5 cluster-split band in shared memory, 6 A load, 7 B
 * load, 8 operand copy source, 9 operand copy destination, 10 reduction
 * input, 11 reduction partial, 12 reduction output). */
const char *gemm_f32_index_site_name(int site);

/*
 * gemm_f32_selftest_index_check -- self-test of the checked build's index
 * checks. Runs gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, mode, kernel,
 * stream) with C declared one row short to the kernels' checks (extent
 * (M - 2) x ldc + N elements instead of (M - 1) x ldc + N), so every store
 * to C's last row fails its check and is skipped: that row keeps its
 * previous contents and gemm_f32_take_index_fault reports a C-store site.
 * Every access it makes stays inside the M x N matrix passed, which must be
 * valid memory as for gemm_f32. Requires M >= 2 and K >= 1; returns what
 * the launch returns, GEMM_ERR_INVALID_ARG for bad arguments and always in
 * the regular build (nothing to check there).
 */
int gemm_f32_selftest_index_check(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                  const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                                  int kernel, void *stream);

/*
 * gemm_f32_selftest_wait_timeout -- failure-detection self-test. Launches one
 * warp that waits, through the same bounded pipeline wait the GEMM kernels
 * use, on a shared-memory barrier that nothing ever signals; after
 * `timeout_ns` (1e6 .. 1e10) the wait gives up, records GEMM_ERR_TIMEOUT in
 * the device status word and the kernel returns. Synchronises `stream` and
 * returns what gemm_f32_poll_device_status then reads (GEMM_ERR_TIMEOUT when
 * the mechanism works). The context stays usable afterwards.
 */
int gemm_f32_selftest_wait_timeout(int64_t timeout_ns, void *stream);

/*
 * gemm_f32_selftest_stalled_gemm -- failure-detection self-test of the GEMM
 * kernels' own abort path. Runs the TMA-fed CTA-pair kernel of `mode`
 * (GEMM_F32_EXACT: 3xTF32; GEMM_F32_TF32: one TF32 pass) on C = A x B with
 * every pipeline wait limited to `timeout_ns` (1e6 .. 1e10), and with its
 * producers stopping after their first k-block: they issue no further copy
 * and no arrival, and wait (bounded) for the copies they did issue, so
 * nothing they started is still in flight. The MMA, transform and epilogue
 * roles then wait for k-blocks that never come; their waits run out, record
 * GEMM_ERR_TIMEOUT in the device status word and raise the CTA's abort flag;
 * every role leaves its loop, the MMAs issued so far complete, both CTAs of
 * each pair meet at the cluster barrier, TMEM is freed and the kernel
 * returns. A problem with few output tiles runs on the cluster-split
 * variant, as gemm_f32 would run it (its CTAs then also skip the sum of the
 * partial tiles and meet at the second cluster barrier). Synchronises
 * `stream` and returns what gemm_f32_poll_device_status then reads
 * (GEMM_ERR_TIMEOUT when the abort path works); C's contents are
 * unspecified afterwards. The context stays usable.
 *   M, N, K, A, lda, B, ldb, C, ldc   as for gemm_f32, with K >= 64 (two
 *             k-blocks), A and B 16-byte aligned with pitches that are
 *             multiples of 4, and a problem whose tiles gemm_f32 would not
 *             split through its workspace (no more unit tiles than CTA
 *             pairs, or few enough for the cluster split), else
 *             GEMM_ERR_INVALID_ARG.
 * The pages have no counterpart: their kernels have no waits that can fail.
 */
int gemm_f32_selftest_stalled_gemm(int64_t M, int64_t N, int64_t K,
                                   const float *A, int64_t lda,
                                   const float *B, int64_t ldb,
                                   float *C, int64_t ldc,
                                   int mode, int64_t timeout_ns, void *stream);

/*
 * gemm_f32_selftest_host_missing_block -- failure-detection self-test of
 * gemm_f32_host's fed launch (exact mode, K >= 16). Runs gemm_f32_host(M, N,
 * K, A, lda, B, ldb, C, ldc, GEMM_F32_EXACT) with every device-side wait
 * limited to `timeout_ns` (1e6 .. 1e10), except that the copy stream never
 * writes the ready word of A's last block (the copy itself still runs). The
 * kernel's waits for those rows run out: they record GEMM_ERR_TIMEOUT, the
 * CTAs give up as in gemm_f32_selftest_stalled_gemm and raise every done
 * counter, so the copies of C go ahead and the call returns. Returns what
 * the call returns (GEMM_ERR_TIMEOUT when the mechanism works; C's contents
 * are then unspecified); GEMM_ERR_INVALID_ARG for bad arguments, K < 16, or
 * a driver without stream memory operations (no fed launch to test). The
 * context stays usable.
 */
int gemm_f32_selftest_host_missing_block(int64_t M, int64_t N, int64_t K,
                                         const float *A, int64_t lda,
                                         const float *B, int64_t ldb,
                                         float *C, int64_t ldc, int64_t timeout_ns);

/* Kinds of tensor-core launch for gemm_f32_schedule_check. */
typedef enum {
    GEMM_SCHEDULE_EXACT_PAIR = 0,  /* 3xTF32 on CTA pairs (TMA-fed, exact mode) */
    GEMM_SCHEDULE_TF32_PAIR = 1,   /* one TF32 pass on CTA pairs (TMA-fed) */
    GEMM_SCHEDULE_EXACT_LSU = 2,   /* 3xTF32 on one SM per tile, plain loads */
    GEMM_SCHEDULE_TF32_LSU = 3     /* one TF32 pass on one SM per tile, plain loads */
} gemm_f32_schedule_kind;

/*
 * gemm_f32_schedule_check -- host-only self-check of the tile scheduler; no
 * GPU or CUDA call. For an M x N x K problem on `workers` clusters (CTA pairs,
 * or SMs for the plain-load kind), builds the schedule the library launches
 * with and walks every cluster's work list with the kernels' own code. It
 * checks that:
 *   - every k-block of every output tile is computed exactly once;
 *   - a whole-tile unit spans the tile's k range;
 *   - the parts of a split tile are numbered 0 .. nparts - 1 in k order, at
 *     most 8 of them;
 *   - each part's partial-sum slot belongs to its own cluster and no slot is
 *     shared;
 *   - for the pair kinds, when there are at most half as many unit tiles as
 *     pairs (the cluster split: 2 to 4 pairs of one cluster take contiguous
 *     k-slices of one unit tile and sum them after a cluster barrier, through
 *     one workspace slot per CTA and no counters), that each pair has
 *     exactly one non-empty slice and the slices of a tile follow each
 *     other in pair order. (On a GPU the
 *     library also lowers the pairs per tile until all the clusters fit on
 *     the device at once, which this host-only check cannot see.)
 *   M, N, K     >= 1 and below 2^31; tiles x k-blocks at most 2^26
 *   workers     1 .. 4096
 *   kind        a gemm_f32_schedule_kind
 *   stats       host array of 9 int64 (written on success): unit tiles,
 *               k-blocks per tile, whole tiles, stream-K share, stream-K
 *               clusters, 1 if some tile is split through the workspace,
 *               most parts of one tile, clusters (pairs or SMs) launched,
 *               pairs per tile in a cluster split (1: none)
 * Returns GEMM_OK; GEMM_ERR_INVALID_ARG for bad arguments; otherwise a code
 * from 10 up that names the check that failed (see its definition).
 */
int gemm_f32_schedule_check(int64_t M, int64_t N, int64_t K, int64_t workers, int kind,
                            int64_t *stats);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F32_H */
