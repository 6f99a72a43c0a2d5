/*
 * ORACLE: test infrastructure, not part of the library.
 *
 * A plain, slow, fp64 CPU statement of the dense projection, used only to
 * check the CUDA path.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code with the CUDA
 * library: its own bf16 decoding, its own loops, no headers in common.
 *
 * What it computes ("How I made Muse's GPU projections 1.32× faster in the
 * Open Kernel Challenge", section "The full equation, now with the letters
 * explained"):
 *
 *     Y[m, n] = Σ_{k=0}^{K-1} X[m, k] · W[n, k]          (+ bias[n])
 *
 * written as the page's plain m / n / k loop, in fp64, over the bf16 inputs
 * decoded exactly.  Every product of two bf16 values is exact in fp64 (8+8
 * significant bits), so the only rounding is fp64 summation in k order.
 *
 * Readings where the pages are silent:
 *  - bias: the page's own task has none (section "What makes it linear?"
 *    calls a matrix product plus a fixed bias an affine map); when present it
 *    is broadcast over token rows and added once, after the K sum.
 *  - the result stays fp64; callers compare a device output decoded to fp64.
 *  - W storage: layout 0 is [N, K] with K contiguous (element (n,k) at
 *    n·K + k, section "What a matrix looks like in memory"); layout 1 is the
 *    copied transpose [K, N] with N contiguous (element (n,k) at k·N + n).
 *
 * OpenMP spreads independent output cells over host threads; each cell's sum
 * is still the single sequential k loop.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* A bf16 value is the upper half of an fp32 bit pattern (1 sign, 8 exponent,
 * 7 fraction bits: section "What a floating-point number is approximating"),
 * so widening is a 16-bit shift; fp32 → fp64 is then exact. */
double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double w_elem(const uint16_t *W, int w_layout, int64_t N, int64_t K,
                     int64_t n, int64_t k) {
    return oracle_bf16_to_double(w_layout == 0 ? W[n * K + k] : W[k * N + n]);
}

/* One output cell: the page's innermost loop. */
static double cell(int64_t N, int64_t K, const uint16_t *X, const uint16_t *W,
                   int w_layout, const uint16_t *bias, int64_t m, int64_t n) {
    double total = 0.0;
    for (int64_t k = 0; k < K; ++k)
        total += oracle_bf16_to_double(X[m * K + k]) * w_elem(W, w_layout, N, K, n, k);
    if (bias)
        total += oracle_bf16_to_double(bias[n]);
    return total;
}

/* Y (fp64, [M, N] row-major) for the whole problem.  bias may be NULL. */
void oracle_project(int64_t M, int64_t N, int64_t K, const uint16_t *X,
                    const uint16_t *W, int w_layout, const uint16_t *bias,
                    double *Y) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] = cell(N, K, X, W, w_layout, bias, m, n);
}

/* The same cells at chosen coordinates (ms[i], ns[i]), i < count. */
void oracle_project_cells(int64_t M, int64_t N, int64_t K, const uint16_t *X,
                          const uint16_t *W, int w_layout, const uint16_t *bias,
                          int64_t count, const int64_t *ms, const int64_t *ns,
                          double *out) {
    (void)M;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = cell(N, K, X, W, w_layout, bias, ms[i], ns[i]);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
