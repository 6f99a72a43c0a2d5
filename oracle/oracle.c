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
#include <math.h>
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

/* ------------------------------------------------------------------------
 * FP32 router weights ("How I made Muse's GPU projections 1.32× faster in the
 * Open Kernel Challenge", section "Why the high-plus-low router scheme
 * helped"): the weight is fp32, and the method keeps a bf16 high part and a
 * bf16 low part of it:
 *
 *     H = roundBF16(W),  R = W − FP32(H),  L = roundBF16(R),  X·Wᵀ ≈ X·Hᵀ + X·Lᵀ.
 *
 * roundBF16 is round to nearest, ties to even (section "What a floating-point
 * number is approximating": bf16 keeps 7 of fp32's 23 fraction bits).  The
 * residual R is an fp32 subtraction, as the section writes it.
 * ------------------------------------------------------------------------ */

/* fp32 → bf16 bits, round to nearest, ties to even.  A NaN stays a (quiet)
 * NaN.  Rounding adds just under half of the dropped 16 bits' range, plus one
 * more when the kept part is odd, then drops them: ties go to even. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t keep_odd = (u >> 16) & 1u;
    u += 0x7FFFu + keep_odd;
    return (uint16_t)(u >> 16);
}

/* H and L for `count` fp32 weights (any layout: element by element). */
void oracle_split_hilo(int64_t count, const float *W, uint16_t *H, uint16_t *L) {
    for (int64_t i = 0; i < count; ++i) {
        const uint16_t h = oracle_f32_to_bf16(W[i]);
        const float h32 = (float)oracle_bf16_to_double(h);
        const float r = W[i] - h32;
        H[i] = h;
        L[i] = oracle_f32_to_bf16(r);
    }
}

/* The router's reference: the exact product with the fp32 weight, in fp64
 * (each bf16 × fp32 product has at most 8 + 24 significant bits: exact). */
static double cell_f32w(int64_t N, int64_t K, const uint16_t *X, const float *W,
                        int w_layout, const uint16_t *bias, int64_t m, int64_t n) {
    double acc = 0.0;
    for (int64_t kk = 0; kk < K; ++kk) {
        const double w = (double)(w_layout == 0 ? W[n * K + kk] : W[kk * N + n]);
        acc += oracle_bf16_to_double(X[m * K + kk]) * w;
    }
    if (bias)
        acc += oracle_bf16_to_double(bias[n]);
    return acc;
}

void oracle_project_f32w(int64_t M, int64_t N, int64_t K, const uint16_t *X,
                         const float *W, int w_layout, const uint16_t *bias,
                         double *Y) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] = cell_f32w(N, K, X, W, w_layout, bias, m, n);
}

/* ------------------------------------------------------------------------
 * Fused epilogues.  The worklog's second page fuses the FFN's activation into
 * the projection's epilogue ("FFN intermediate written, re-read for GELU,
 * written again" → written once), and a residual connection adds an earlier
 * representation back to the projected one (first page, section
 * "Normalization and residuals also cost time").  The pages do not write the
 * activation out; this oracle takes GELU's definition, x·Φ(x) with Φ the
 * standard normal CDF: GELU(x) = x/2 · (1 + erf(x/√2)).
 * ------------------------------------------------------------------------ */
double oracle_gelu(double x) {
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

/* SwiGLU's gate nonlinearity (Shazeer, "GLU Variants Improve Transformer",
 * 2020): SiLU(x) = x · σ(x) = x / (1 + e^(−x)).  The first page's
 * section on experts combines two projections of one input entry by entry,
 * one of them passed through a nonlinearity it does not name; SwiGLU names
 * it. */
double oracle_silu(double x) {
    return x / (1.0 + exp(-x));
}

/* SwiGLU of a gate and an up array: out[i] = SiLU(gate[i]) · up[i]. */
void oracle_swiglu(int64_t count, const double *gate, const double *up, double *out) {
    for (int64_t i = 0; i < count; ++i) out[i] = oracle_silu(gate[i]) * up[i];
}

/* In place over `count` values: act 0 = identity, 1 = GELU. */
void oracle_apply_activation(int64_t count, int act, double *v) {
    if (act == 1)
        for (int64_t i = 0; i < count; ++i) v[i] = oracle_gelu(v[i]);
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
