/*
 * fp64 oracle for the sum of a vector of single-precision values.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *
 *     s64 = sum_{i = 0 .. n-1} (double)x[i]      S = sum_{i} |x[i]|
 *
 * in increasing i. This is the quantity that the reduction of "GPU compute
 * shaders" ("How it works", step 6, and the reduce routine under "Code")
 * computes with per-group partial sums combined in a second dispatch; the
 * page's own check compares it against a plain sequential sum.
 *
 * Precision: each fp32 value is exact in fp64 and the fp64 accumulation
 * adds at most about n 2^-53 S of error, negligible next to any fp32 bound
 * for the sizes used here. The build disables floating-point contraction.
 */
#include <math.h>
#include <stdint.h>

void oracle_sum_f64(int64_t n, const float *x, double *s64, double *S)
{
    double acc = 0.0, scale = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double v = (double)x[i];
        acc += v;
        scale += fabs(v);
    }
    *s64 = acc;
    if (S) *S = scale;
}
