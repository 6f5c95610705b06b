/*
 * dg_oracle.c -- plain, slow, fp64 CPU reference for the decode-time skinny linears.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or constant with the CUDA path, and it never calls it.
 *
 * What it follows (pages cited by title and section):
 *   - decode linears y = x.W^T at 1-128 rows, the fused gate/up entry with
 *     SiLU.mul: mstar PR #1104 (decode GEMM table), "Why" and "What changed";
 *   - the fp8 vocabulary head with one scale for the whole head, and greedy
 *     (temperature 0) sampling of its logits: mstar PR #1102 (fused draft step
 *     and fp8 draft head), "What changed";
 *   - routed MoE experts with W1/W2 at small token counts: "Decode optimization
 *     round 3", "Retained change 1: N-split W1/W2 MoE kernels".
 * The pages print no formulas; each function below states the plain
 * definition it computes.  Every sum runs in plain ascending k order in
 * double precision; OpenMP only splits independent outputs across threads.
 * Build with -ffp-contract=off so that x86 and Arm give identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DGO_API __attribute__((visibility("default")))

/* bf16 is the upper 16 bits of an IEEE binary32 value. */
static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit float E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent field 0 encodes subnormals m * 2^-9; no infinities;
 * S.1111.111 is NaN; the largest finite magnitude is 448. */
DGO_API double dgo_e4m3_value(uint8_t q)
{
    const int sign = (q >> 7) & 1;
    const int expo = (q >> 3) & 0xF;
    const int mant = q & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    switch (expo) {
    case 0:
        mag = ldexp((double)mant, -9);
        break;
    default:
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
        break;
    }
    return sign ? -mag : mag;
}

/* The same values as a 256-entry table, filled from dgo_e4m3_value once (speed only). */
static double e4m3_table[256];
static int e4m3_table_ready = 0;

static void e4m3_table_init(void)
{
    if (e4m3_table_ready)
        return;
    for (int c = 0; c < 256; ++c)
        e4m3_table[c] = dgo_e4m3_value((uint8_t)c);
    e4m3_table_ready = 1;
}

#define E4M3(c) (e4m3_table[(c)])

/* Round a double to the nearest bf16 (ties to even), directly from the double
 * (no detour through binary32, which could round twice). */
static uint16_t round_to_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                /* quantum of an 8-significant-bit value */
    if (q < -133)
        q = -133;                 /* bf16 subnormal spacing 2^-133 */
    double r = nearbyint(ldexp(a, -q));   /* default rounding mode: ties to even */
    double out = ldexp(r, q);
    if (out >= 0x1p128)
        return sign | 0x7F80;     /* overflow to infinity */
    float f = (float)out;         /* exact: out has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

DGO_API void dgo_round_bf16(const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = round_to_bf16(in[i]);
}

DGO_API void dgo_bf16_to_double(const uint16_t* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_value(in[i]);
}

static int64_t pick_row(const int64_t* rows, int64_t r) { return rows ? rows[r] : r; }

/* Linear: y[m, r] = sum_k x[m,k] * W[n_r, k] for the requested rows n_r (all rows
 * when rows == NULL, nrows = N).  absdot[m, r] = sum_k |x[m,k] * W[n_r,k]| feeds the
 * error bound.  x [M,K] and W [N,K] are bf16 bit patterns, row-major. */
DGO_API void dgo_linear_bf16(const uint16_t* x, const uint16_t* W, int64_t M, int64_t K,
                             const int64_t* rows, int64_t nrows, double* y, double* absdot)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint16_t* w = W + pick_row(rows, r) * K;
        for (int64_t m = 0; m < M; ++m) {
            const uint16_t* xm = x + m * K;
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = bf16_value(xm[k]) * bf16_value(w[k]);
                s += p;
                a += fabs(p);
            }
            y[m * nrows + r] = s;
            if (absdot)
                absdot[m * nrows + r] = a;
        }
    }
}

/* SiLU (swish with unit slope): silu(g) = g * sigmoid(g) = g / (1 + exp(-g)). */
DGO_API double dgo_silu(double g) { return g / (1.0 + exp(-g)); }

/* Fused gate/up: W_gu is [2*Nh, K] with gate row j at 2j and up row j at 2j+1.
 * For each requested output column j: g = x.W_gu[2j], u = x.W_gu[2j+1],
 * out[m, c] = silu(g) * u.  g, u, sum|x*w_gate|, sum|x*w_up| are returned too. */
DGO_API void dgo_gate_up_silu(const uint16_t* x, const uint16_t* Wgu, int64_t M, int64_t K,
                              const int64_t* cols, int64_t ncols, double* out, double* g_out,
                              double* u_out, double* absg, double* absu)
{
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < ncols; ++c) {
        const int64_t j = pick_row(cols, c);
        const uint16_t* wg = Wgu + (2 * j) * K;
        const uint16_t* wu = Wgu + (2 * j + 1) * K;
        for (int64_t m = 0; m < M; ++m) {
            const uint16_t* xm = x + m * K;
            double g = 0.0, u = 0.0, ag = 0.0, au = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double xv = bf16_value(xm[k]);
                const double pg = xv * bf16_value(wg[k]);
                const double pu = xv * bf16_value(wu[k]);
                g += pg;
                u += pu;
                ag += fabs(pg);
                au += fabs(pu);
            }
            const int64_t o = m * ncols + c;
            out[o] = dgo_silu(g) * u;
            if (g_out) g_out[o] = g;
            if (u_out) u_out[o] = u;
            if (absg) absg[o] = ag;
            if (absu) absu[o] = au;
        }
    }
}

/* fp8 head: logit[m, r] = scale * sum_k x[m,k] * e4m3(Wq[n_r, k]) (one scale for
 * the whole matrix).  absdot = |scale| * sum_k |x * e4m3(w)|. */
DGO_API void dgo_head_fp8(const uint16_t* x, const uint8_t* Wq, double scale, int64_t M, int64_t K,
                          const int64_t* rows, int64_t nrows, double* logit, double* absdot)
{
    e4m3_table_init();
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const uint8_t* w = Wq + pick_row(rows, r) * K;
        for (int64_t m = 0; m < M; ++m) {
            const uint16_t* xm = x + m * K;
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = bf16_value(xm[k]) * E4M3(w[k]);
                s += p;
                a += fabs(p);
            }
            logit[m * nrows + r] = scale * s;
            if (absdot)
                absdot[m * nrows + r] = fabs(scale) * a;
        }
    }
}

/* Greedy pick over the whole head: idx[m] = the lowest n whose logit, rounded to
 * binary32 (the precision the pick is taken in), is the largest.  NaN logits are
 * never picked; a row of only NaN gives -1.  best[m] is that binary32 logit and
 * gap[m] = best - (largest logit at any other index, in double) for near-tie checks. */
DGO_API void dgo_head_argmax(const uint16_t* x, const uint8_t* Wq, double scale, int64_t M,
                             int64_t N, int64_t K, int32_t* idx, float* best, double* gap)
{
    double* lg = (double*)malloc(sizeof(double) * (size_t)N * (size_t)M);
    if (!lg)
        return;
    dgo_head_fp8(x, Wq, scale, M, K, NULL, N, lg, NULL);
    for (int64_t m = 0; m < M; ++m) {
        const double* l = lg + m * N;
        int64_t bi = -1;
        float bv = 0.0f;
        for (int64_t n = 0; n < N; ++n) {
            const float v = (float)l[n];
            if (isnan(v))
                continue;
            if (bi < 0 || v > bv) {
                bi = n;
                bv = v;
            }
        }
        idx[m] = (int32_t)bi;
        best[m] = bv;
        if (gap) {
            double second = -INFINITY;
            for (int64_t n = 0; n < N; ++n)
                if (n != bi && !isnan(l[n]) && l[n] > second)
                    second = l[n];
            gap[m] = bi < 0 ? 0.0 : l[bi] - second;
        }
    }
    free(lg);
}

/* MoE routing.  A slot (t, k) is valid when 0 <= ids[t,k] < E and no earlier slot
 * of token t names the same expert.  Outputs:
 *   valid[t*topk + k]          1 / 0
 *   experts[0..U-1]            the active experts in ascending order (returns U)
 *   offsets[0..U]              pairs of active expert u are pairs[offsets[u]..offsets[u+1])
 *   pair_tok / pair_slot       the (token, slot) pairs, ascending by token then slot. */
DGO_API int32_t dgo_moe_route(const int32_t* ids, int64_t M, int64_t topk, int64_t E,
                              int32_t* valid, int32_t* experts, int32_t* offsets,
                              int32_t* pair_tok, int32_t* pair_slot)
{
    for (int64_t t = 0; t < M; ++t)
        for (int64_t k = 0; k < topk; ++k) {
            const int32_t e = ids[t * topk + k];
            int ok = (e >= 0 && e < E);
            for (int64_t j = 0; ok && j < k; ++j)
                if (ids[t * topk + j] == e)
                    ok = 0;
            valid[t * topk + k] = ok;
        }
    int32_t U = 0, P = 0;
    for (int64_t e = 0; e < E; ++e) {
        int32_t start = P;
        for (int64_t t = 0; t < M; ++t)
            for (int64_t k = 0; k < topk; ++k)
                if (valid[t * topk + k] && ids[t * topk + k] == e) {
                    pair_tok[P] = (int32_t)t;
                    pair_slot[P] = (int32_t)k;
                    ++P;
                }
        if (P > start) {
            experts[U] = (int32_t)e;
            offsets[U] = start;
            ++U;
        }
    }
    offsets[U] = P;
    return U;
}

/* MoE W1 + SiLU.mul.  W1 [E, 2I, K] e4m3 codes (rows 0..I-1 gate, I..2I-1 up), s1
 * [E, 2I] one scale per row.  For each valid slot (t,k), e = ids[t,k], j < I:
 *   g = s1[e,j]   * sum_k x[t,:] * e4m3(W1[e, j, :])
 *   u = s1[e,I+j] * sum_k x[t,:] * e4m3(W1[e, I+j, :])
 *   a[t,k,j] = silu(g) * u;   invalid slots give a = 0.
 * absg/absu = |s| * sum |x * w| of the two rows (error bounds); any may be NULL. */
DGO_API void dgo_moe_w1_silu(const uint16_t* x, const int32_t* ids, const uint8_t* W1,
                             const float* s1, int64_t M, int64_t topk, int64_t E, int64_t I,
                             int64_t K, double* a, double* g_out, double* u_out, double* absg,
                             double* absu)
{
    e4m3_table_init();
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < M; ++t)
        for (int64_t k = 0; k < topk; ++k) {
            const int32_t e = ids[t * topk + k];
            int ok = (e >= 0 && e < E);
            for (int64_t j = 0; ok && j < k; ++j)
                if (ids[t * topk + j] == e)
                    ok = 0;
            for (int64_t j = 0; j < I; ++j) {
                const int64_t o = (t * topk + k) * I + j;
                if (!ok) {
                    a[o] = 0.0;
                    if (g_out) g_out[o] = 0.0;
                    if (u_out) u_out[o] = 0.0;
                    if (absg) absg[o] = 0.0;
                    if (absu) absu[o] = 0.0;
                    continue;
                }
                const uint8_t* wg = W1 + ((int64_t)e * 2 * I + j) * K;
                const uint8_t* wu = W1 + ((int64_t)e * 2 * I + I + j) * K;
                const double sg = s1[(int64_t)e * 2 * I + j];
                const double su = s1[(int64_t)e * 2 * I + I + j];
                double g = 0.0, u = 0.0, ag = 0.0, au = 0.0;
                for (int64_t kk = 0; kk < K; ++kk) {
                    const double xv = bf16_value(x[t * K + kk]);
                    const double pg = xv * E4M3(wg[kk]);
                    const double pu = xv * E4M3(wu[kk]);
                    g += pg;
                    u += pu;
                    ag += fabs(pg);
                    au += fabs(pu);
                }
                g *= sg;
                u *= su;
                a[o] = dgo_silu(g) * u;
                if (g_out) g_out[o] = g;
                if (u_out) u_out[o] = u;
                if (absg) absg[o] = fabs(sg) * ag;
                if (absu) absu[o] = fabs(su) * au;
            }
        }
}

/* MoE W2 + weighted combine.  a [M, topk, I] bf16 (the activations that W2 reads),
 * W2 [E, Nout, I] e4m3 codes, s2 [E, Nout], gate weights gw [M, topk] fp32:
 *   y[t, n] = sum over valid slots k of gw[t,k] * s2[e,n] * sum_i a[t,k,i] * e4m3(W2[e,n,i])
 * absdot[t, n] = sum over valid k of |gw * s2| * sum_i |a * w|. */
DGO_API void dgo_moe_w2(const uint16_t* a, const int32_t* ids, const float* gw, const uint8_t* W2,
                        const float* s2, int64_t M, int64_t topk, int64_t E, int64_t I,
                        int64_t Nout, double* y, double* absdot)
{
    e4m3_table_init();
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < M; ++t)
        for (int64_t n = 0; n < Nout; ++n) {
            double acc = 0.0, bound = 0.0;
            for (int64_t k = 0; k < topk; ++k) {
                const int32_t e = ids[t * topk + k];
                int ok = (e >= 0 && e < E);
                for (int64_t j = 0; ok && j < k; ++j)
                    if (ids[t * topk + j] == e)
                        ok = 0;
                if (!ok)
                    continue;
                const uint8_t* w = W2 + ((int64_t)e * Nout + n) * I;
                const uint16_t* at = a + (t * topk + k) * I;
                double h = 0.0, ah = 0.0;
                for (int64_t i = 0; i < I; ++i) {
                    const double p = bf16_value(at[i]) * E4M3(w[i]);
                    h += p;
                    ah += fabs(p);
                }
                const double c = (double)gw[t * topk + k] * (double)s2[(int64_t)e * Nout + n];
                acc += c * h;
                bound += fabs(c) * ah;
            }
            y[t * Nout + n] = acc;
            if (absdot)
                absdot[t * Nout + n] = bound;
        }
}

/* ---------------------------------------------------------------- A8W8 blockscale
 * The A8W8 block-scaled linear and the activation quantisation it takes as a
 * prologue ("Decode optimization round 3", "Retained change 2: decode-M rows for
 * the A8W8 bpreshuffle table", and "Rejected paths" / "Remaining headroom": the
 * quantisation kernels fused into the GEMM).  Blocks are 128 wide along K: one
 * activation scale per (token, K-block), one weight scale per 128 x 128 block.
 * The pages give no formulas; the quantisation below is the plain per-block
 * max-scaling to the e4m3 range, decided in binary32. */

/* Nearest e4m3 code to a binary32 value, ties to even, magnitudes beyond 448
 * clamped to 448 (saturating), NaN to 0x7F.  Written from the field layout:
 * normal values (1 + m/8) * 2^(e-7) for biased exponent e = 1..15, subnormals
 * m * 2^-9. */
DGO_API uint8_t dgo_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < 0x1p-6) {                                   /* subnormal range, spacing 2^-9 */
        const double m = nearbyint(a * 0x1p9);         /* 0 .. 8; 8 is the smallest normal */
        return sign | (uint8_t)m;
    }
    int e;
    frexp(a, &e);                                       /* a = f * 2^e, f in [0.5, 1) */
    const int unbiased = e - 1;                         /* a = (1 + m/8) * 2^unbiased */
    double m = nearbyint(ldexp(a, 3 - unbiased)) - 8.0; /* 0 .. 8 */
    int ub = unbiased;
    if (m >= 8.0) {
        m = 0.0;
        ++ub;
    }
    if (ub + 7 > 15 || (ub + 7 == 15 && m > 6.0))     /* above 448 after rounding */
        return sign | 0x7E;
    return sign | (uint8_t)(((ub + 7) << 3) | (int)m);
}

/* Per token m and K-block b (elements b*128 .. min(K, b*128+128) - 1), in binary32:
 *   amax = max(max |x|, 2^-32)      (all-zero blocks quantise to zero codes)
 *   r    = 448 / amax               sx[m, b] = amax / 448
 *   q[m, k] = e4m3(x[m, k] * r)
 * x [M, K] bf16 bits; q [M, K] codes; sx [M, ceil(K/128)]. */
DGO_API void dgo_a8_quant(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, float* sx)
{
    const int64_t nb = (K + 127) / 128;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            const int64_t k0 = b * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
            float amax = 0.0f;
            for (int64_t k = k0; k < k1; ++k) {
                const float a = fabsf((float)bf16_value(x[m * K + k]));
                if (a > amax)
                    amax = a;
            }
            if (amax < 0x1p-32f)
                amax = 0x1p-32f;
            const float r = 448.0f / amax;
            sx[m * nb + b] = amax / 448.0f;
            for (int64_t k = k0; k < k1; ++k) {
                const float v = (float)bf16_value(x[m * K + k]) * r;
                q[m * K + k] = dgo_e4m3_encode(v);
            }
        }
}

/* y[m, r] = sum over K-blocks b of sx[m,b] * sw[n/128, b] * sum_{k in b} e4m3(q[m,k]) *
 * e4m3(Wq[n,k]) for the requested rows n = n_r, in double (every product and the
 * block sums are exact there; the blocks are added in ascending b).
 * absdot[m, r] = sum_b |sx * sw| * sum_k |q * w|.  Wq [N, K] codes,
 * sw [ceil(N/128), ceil(K/128)] fp32 row-major. */
DGO_API void dgo_a8w8_linear(const uint8_t* q, const float* sx, const uint8_t* Wq, const float* sw,
                             int64_t M, int64_t K, const int64_t* rows, int64_t nrows, double* y,
                             double* absdot)
{
    e4m3_table_init();
    const int64_t nb = (K + 127) / 128;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t n = pick_row(rows, r);
        const uint8_t* w = Wq + n * K;
        for (int64_t m = 0; m < M; ++m) {
            double s = 0.0, a = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const int64_t k0 = b * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
                double d = 0.0, ad = 0.0;
                for (int64_t k = k0; k < k1; ++k) {
                    const double p = E4M3(q[m * K + k]) * E4M3(w[k]);
                    d += p;
                    ad += fabs(p);
                }
                const double c = (double)sx[m * nb + b] * (double)sw[(n / 128) * nb + b];
                s += c * d;
                a += fabs(c) * ad;
            }
            y[m * nrows + r] = s;
            if (absdot)
                absdot[m * nrows + r] = a;
        }
    }
}
