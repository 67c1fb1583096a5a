/*
 * reduce_f32.h -- C ABI of libgemm_f32.so, part 2: the sum of a fp32 vector
 * on an NVIDIA GB300 (sm_103a).
 *
 * Operation. out[0] = sum_{i < n} x[i], computed as in "GPU compute shaders"
 * ("How it works", step 6, and the reduce routine under "Code"): `groups`
 * groups each walk x with a grid stride and reduce their threads' sums by a
 * tree to one partial sum; a second dispatch adds the partials. Status codes
 * are those of gemm_f32.h.
 *
 * Determinism: for the same n, groups, device and 16-byte alignment of x,
 * every addition happens in the same order, so reruns give bit-identical
 * results (the page's "Pitfalls": a float sum is reproducible only when the
 * group count and the order are fixed).
 *
 * Accuracy: with G groups, |out - sum x| <= h 2^-24 sum |x| (to first order),
 * h = ceil(n / (1024 G)) + ceil(G / 256) + 24: each element passes through at
 * most h fp32 roundings.
 */
#ifndef REDUCE_F32_H
#define REDUCE_F32_H

#include <stdint.h>

#include "gemm_f32.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * reduce_f32_sum -- *out = sum of x[0, n), stream ordered.
 *   n       elements, 0 <= n <= 2^40; n == 0 sets *out = 0.
 *   x       device pointer to n fp32 values, 4-byte aligned (16-byte aligned
 *           x takes 128-bit loads).
 *   out     device pointer to one fp32, 4-byte aligned, outside x
 *           (GEMM_ERR_ALIAS otherwise).
 *   groups  number of partial sums, 1 .. 65535, or 0 for the default (four
 *           per SM). It fixes the summation order.
 *   stream  cudaStream_t as void* (NULL = the legacy default stream).
 * The partial sums live in a workspace of `groups` floats taken from the
 * library's stream-ordered memory pool on `stream` and returned behind the
 * second kernel. Argument errors are reported before anything is enqueued.
 * Returns a gemm_f32_status.
 */
int reduce_f32_sum(int64_t n, const float *x, float *out, int groups, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* REDUCE_F32_H */
