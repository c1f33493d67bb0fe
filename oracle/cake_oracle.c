/*
 * cake_oracle.c -- FP64 CPU oracle for the ragged BF16 grouped GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA path is checked against.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library's product
 * path never calls, links or includes anything here, and this file includes
 * nothing from the library.
 *
 * What is computed (flashinfer PR #8258 "perf(cake_moe_grouped_gemm): run the
 * split k512 wgrad tail whole on the least-loaded clusters", opening summary:
 * forward Y = X W^T, data gradient dX = G W, weight gradient dW = G^T X, all
 * with BF16 inputs), per expert e owning the rows [off[e], off[e+1]):
 *
 *   Y [r, n]   = sum_{k <  K}  X[r, k] * W[e, n, k]           (forward)
 *   dX[r, k]   = sum_{n <  N}  G[r, n] * W[e, n, k]           (data gradient)
 *   dW[e, n, k]= sum_{r = off[e]}^{off[e+1]-1} G[r, n] * X[r, k]  (weight gradient)
 *
 * Storage is row-major with the last index contiguous: X [M, K], W [E, N, K],
 * G [M, N], Y [M, N], dX [M, K], dW [E, N, K].  This is the nn.Linear layout
 * implied by Y = X W^T, and matches the dense projection page's layouts
 * (flashinfer PR #8363, "Definitions": activations [T, d_in], output
 * gradients [T, d_out], weight gradient [d_out, d_in]).
 *
 * Arithmetic: every BF16 value is widened exactly to double; each output is a
 * sequential FP64 sum in increasing index order; the result is returned in
 * FP64 and never rounded.  Rows at or beyond off[E] are not computed.  An
 * empty expert (off[e] == off[e+1]) has an exact zero weight gradient.
 * Parallelism (OpenMP over independent outputs) never changes the order of
 * any one sum.
 *
 * Every entry point validates the offsets (off[0] == 0, non-decreasing,
 * off[E] <= M) and returns 0 on success, -1 on invalid arguments.
 *
 * The FP32 router GEMM of the same family (BF16x3 emulation) is at the end of
 * this file.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake; it is
 * used only by the test that shows the oracle's pins catch such mistakes.
 */
#include <stdint.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* Exact widening: a BF16 value is the top half of an IEEE binary32. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int offsets_ok(const int32_t *off, int32_t E, int64_t M)
{
    if (E < 1 || off == 0) return 0;
    if (off[0] != 0) return 0;
    for (int32_t e = 0; e < E; ++e)
        if (off[e + 1] < off[e]) return 0;
    return (int64_t)off[E] <= M;
}

/* Expert owning row r (r < off[E]); the last e with off[e] <= r < off[e+1]. */
static int32_t expert_of_row(const int32_t *off, int32_t E, int64_t r)
{
    int32_t lo = 0, hi = E - 1;
    while (lo < hi) {
        int32_t mid = (lo + hi + 1) / 2;
        if ((int64_t)off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* ---- one output element of each pass ---------------------------------- */

static double fwd_elem(const uint16_t *X, const uint16_t *W, int32_t e, int64_t r,
                       int32_t n, int32_t N, int32_t K)
{
    const uint16_t *x = X + r * (int64_t)K;
    const uint16_t *w = W + ((int64_t)e * N + n) * (int64_t)K;
    double s = 0.0;
    for (int32_t k = 0; k < K; ++k) {
#if ORACLE_MUTANT == 1 /* planted mistake: one term of the sum dropped */
        if (k == K - 1) break;
#endif
        s += bf16_to_f64(x[k]) * bf16_to_f64(w[k]);
    }
    return s;
}

static double dgrad_elem(const uint16_t *G, const uint16_t *W, int32_t e, int64_t r,
                         int32_t k, int32_t N, int32_t K)
{
    const uint16_t *g = G + r * (int64_t)N;
    const uint16_t *w = W + (int64_t)e * N * (int64_t)K + k;
    double s = 0.0;
    for (int32_t n = 0; n < N; ++n) {
#if ORACLE_MUTANT == 2 /* planted mistake: W_e read as if stored [K, N] (transposed operand) */
        s += bf16_to_f64(g[n]) * bf16_to_f64(W[(int64_t)e * N * K + (int64_t)k * N + n]);
        continue;
#endif
#if ORACLE_MUTANT == 5 /* planted mistake: wrong sign on the first term */
        if (n == 0) { s -= bf16_to_f64(g[n]) * bf16_to_f64(w[0]); continue; }
#endif
        s += bf16_to_f64(g[n]) * bf16_to_f64(w[(int64_t)n * K]);
    }
    return s;
}

static double wgrad_elem(const uint16_t *G, const uint16_t *X, const int32_t *off,
                         int32_t e, int32_t n, int32_t k, int32_t N, int32_t K)
{
    double s = 0.0;
    int64_t r0 = off[e], r1 = off[e + 1];
#if ORACLE_MUTANT == 3 /* planted mistake: the reduction runs one row past the expert */
    r1 += 1;
#endif
    for (int64_t r = r0; r < r1; ++r)
        s += bf16_to_f64(G[r * N + n]) * bf16_to_f64(X[r * K + k]);
    return s;
}

/* ---- whole-tensor entry points ----------------------------------------- */

/* Y [off[E], N] (FP64), rows >= off[E] untouched. */
int oracle_fwd(const uint16_t *X, const uint16_t *W, const int32_t *off, int32_t E,
               int64_t M, int32_t N, int32_t K, double *Y)
{
    if (!offsets_ok(off, E, M) || N < 1 || K < 1) return -1;
    const int64_t rows = off[E];
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int32_t e = expert_of_row(off, E, r);
#if ORACLE_MUTANT == 4 /* planted mistake: the previous expert's weights */
        if (e > 0) e -= 1;
#endif
        for (int32_t n = 0; n < N; ++n)
            Y[r * N + n] = fwd_elem(X, W, e, r, n, N, K);
    }
    return 0;
}

/* dX [off[E], K] (FP64). */
int oracle_dgrad(const uint16_t *G, const uint16_t *W, const int32_t *off, int32_t E,
                 int64_t M, int32_t N, int32_t K, double *dX)
{
    if (!offsets_ok(off, E, M) || N < 1 || K < 1) return -1;
    const int64_t rows = off[E];
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int32_t e = expert_of_row(off, E, r);
        for (int32_t k = 0; k < K; ++k)
            dX[r * K + k] = dgrad_elem(G, W, e, r, k, N, K);
    }
    return 0;
}

/* dW [E, N, K] (FP64); an empty expert gets exact zeros. */
int oracle_wgrad(const uint16_t *G, const uint16_t *X, const int32_t *off, int32_t E,
                 int64_t M, int32_t N, int32_t K, double *dW)
{
    if (!offsets_ok(off, E, M) || N < 1 || K < 1) return -1;
    const int64_t total = (int64_t)E * N;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t en = 0; en < total; ++en) {
        int32_t e = (int32_t)(en / N), n = (int32_t)(en % N);
        for (int32_t k = 0; k < K; ++k)
            dW[en * K + k] = wgrad_elem(G, X, off, e, n, k, N, K);
    }
    return 0;
}

/* ---- sampled entry points (any size; one element at a time) ------------ */

/* out[i] = Y[rows[i], cols[i]]; every rows[i] must be < off[E]. */
int oracle_fwd_at(const uint16_t *X, const uint16_t *W, const int32_t *off, int32_t E,
                  int64_t M, int32_t N, int32_t K, const int64_t *rows,
                  const int64_t *cols, int64_t count, double *out)
{
    if (!offsets_ok(off, E, M) || N < 1 || K < 1) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= off[E] || cols[i] < 0 || cols[i] >= N) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i)
        out[i] = fwd_elem(X, W, expert_of_row(off, E, rows[i]), rows[i], (int32_t)cols[i], N, K);
    return 0;
}

/* out[i] = dX[rows[i], cols[i]]. */
int oracle_dgrad_at(const uint16_t *G, const uint16_t *W, const int32_t *off, int32_t E,
                    int64_t M, int32_t N, int32_t K, const int64_t *rows,
                    const int64_t *cols, int64_t count, double *out)
{
    if (!offsets_ok(off, E, M) || N < 1 || K < 1) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (rows[i] < 0 || rows[i] >= off[E] || cols[i] < 0 || cols[i] >= K) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i)
        out[i] = dgrad_elem(G, W, expert_of_row(off, E, rows[i]), rows[i], (int32_t)cols[i], N, K);
    return 0;
}

/* out[i] = dW[es[i], ns[i], ks[i]]. */
int oracle_wgrad_at(const uint16_t *G, const uint16_t *X, const int32_t *off, int32_t E,
                    int64_t M, int32_t N, int32_t K, const int64_t *es, const int64_t *ns,
                    const int64_t *ks, int64_t count, double *out)
{
    if (!offsets_ok(off, E, M) || N < 1 || K < 1) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (es[i] < 0 || es[i] >= E || ns[i] < 0 || ns[i] >= N || ks[i] < 0 || ks[i] >= K)
            return -1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < count; ++i)
        out[i] = wgrad_elem(G, X, off, (int32_t)es[i], (int32_t)ns[i], (int32_t)ks[i], N, K);
    return 0;
}

/* ---- FP32 router GEMM (BF16x3 emulation) -------------------------------
 *
 * The dense projection family's FP32 router GEMM (flashinfer PR #8438,
 * "Summary", which names a router GEMM over 256 experts in FP32 emulated
 * with three BF16 products): logits Y [T, R] = X [T, K] W^T with FP32 X and router weights W [R, K].
 * The pages name the emulation and nothing more; the reading taken here is
 * the usual one: every FP32 value v is split as hi = bf16(v) (round to
 * nearest, ties to even) and lo = bf16(v - hi), and the product keeps the
 * three leading terms of (x_hi + x_lo)(w_hi + w_lo):
 *
 *   Y[t, r] ~= sum_k  x_hi w_hi + x_hi w_lo + x_lo w_hi          (x = X[t,k], w = W[r,k])
 *
 * oracle_router_bf16x3 computes exactly that sum in FP64 (each term exact,
 * summed in k order, the three terms of one k in the order written);
 * oracle_router_exact computes the definition sum_k x w in FP64. */

/* Round an FP32 value to the nearest BF16 (ties to even), returned widened
 * to FP32; NaN stays NaN.  Written from the definition: keep the top 16 bits
 * of the binary32 pattern after adding half a BF16 unit in the last place,
 * minus one when the kept part is even (so exact halves go to even). */
static float round_bf16(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u) return v;  /* NaN */
    const uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + keep_lsb;
    u &= 0xFFFF0000u;
    float r;
    memcpy(&r, &u, sizeof r);
    return r;
}

static void split_bf16x2(float v, double *hi, double *lo)
{
    const float h = round_bf16(v);
#if ORACLE_MUTANT == 6 /* planted mistake: the low part is never formed */
    *hi = (double)h;
    *lo = 0.0;
    return;
#endif
    const float l = round_bf16(v - h);   /* v - h is exact in FP32 */
    *hi = (double)h;
    *lo = (double)l;
}

static double router_bf16x3_elem(const float *X, const float *W, int64_t t, int32_t r, int32_t K)
{
    const float *x = X + t * (int64_t)K;
    const float *w = W + (int64_t)r * K;
    double s = 0.0;
    for (int32_t k = 0; k < K; ++k) {
        double xh, xl, wh, wl;
        split_bf16x2(x[k], &xh, &xl);
        split_bf16x2(w[k], &wh, &wl);
        s += xh * wh;
        s += xh * wl;
        s += xl * wh;
    }
    return s;
}

static double router_exact_elem(const float *X, const float *W, int64_t t, int32_t r, int32_t K)
{
    const float *x = X + t * (int64_t)K;
    const float *w = W + (int64_t)r * K;
    double s = 0.0;
    for (int32_t k = 0; k < K; ++k) s += (double)x[k] * (double)w[k];
    return s;
}

/* Y [T, R] (FP64) by the BF16x3 emulation; 0 on success, -1 on bad sizes. */
int oracle_router_bf16x3(const float *X, const float *W, int64_t T, int32_t R, int32_t K, double *Y)
{
    if (T < 0 || R < 1 || K < 1) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int32_t r = 0; r < R; ++r) Y[t * R + r] = router_bf16x3_elem(X, W, t, r, K);
    return 0;
}

/* Y [T, R] (FP64) by the definition sum_k x w. */
int oracle_router_exact(const float *X, const float *W, int64_t T, int32_t R, int32_t K, double *Y)
{
    if (T < 0 || R < 1 || K < 1) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int32_t r = 0; r < R; ++r) Y[t * R + r] = router_exact_elem(X, W, t, r, K);
    return 0;
}

/* out[i] = Y[ts[i], rs[i]] by the BF16x3 emulation (any size). */
int oracle_router_bf16x3_at(const float *X, const float *W, int64_t T, int32_t R, int32_t K,
                            const int64_t *ts, const int64_t *rs, int64_t count, double *out)
{
    if (T < 0 || R < 1 || K < 1) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (ts[i] < 0 || ts[i] >= T || rs[i] < 0 || rs[i] >= R) return -1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) out[i] = router_bf16x3_elem(X, W, ts[i], (int32_t)rs[i], K);
    return 0;
}

/* BF16 rounding of one FP32 value, exposed for the pins. */
float oracle_round_bf16(float v) { return round_bf16(v); }

/* Number of OpenMP threads the entry points above use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
