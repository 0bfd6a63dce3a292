/*
 * amsim_oracle.c -- plain, slow, CPU reference for LUT-simulated approximate
 * floating-point multiplication inside DNN contractions.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links or calls
 * this file; only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg load it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * Source followed: "ApproxTrain: Fast Simulation of Approximate Multipliers
 * for DNN Training and Inference" (arXiv 2209.04161):
 *   - Sec. V-A, Algorithm 1 (mantissa-product LUT generation, carry detection,
 *     4-byte entries holding carry and mantissa, footnote 2);
 *   - Sec. V-B, Algorithm 2 (AMSim: sign XOR, concatenated-mantissa index,
 *     zero when the biased exponent is not above zero or an input is zero,
 *     infinity at or above 255, exponent adjusted by the carry);
 *   - Sec. VI-B, Algorithms 3/4 and Fig. 8 (Conv2D forward, weight gradient,
 *     preceding-layer gradient as IM2COL + GEMM; here written as the direct
 *     sums those GEMMs compute).
 * The Mitchell multiplier (MIT16 in Sec. V-C / Table II) is the logarithmic
 * multiplier: mantissa product 1+x+y when x+y<1, otherwise 2(x+y).
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   operand mantissas are truncated to their top M bits; denormal inputs are
 *   treated as zero; NaN in -> NaN out (canonical 0x7FC00000); Inf times a
 *   zero/denormal -> NaN; Inf times anything else -> signed Inf; the zero test
 *   on the biased exponent comes before the carry adjustment (page order);
 *   an exponent that reaches 255 only through the carry also gives Inf; zero
 *   and Inf results carry the XOR sign; the LUT mantissa is used at its full
 *   23 bits.  Contractions sum the fp32 products in double in natural k order
 *   and round once; padding / non-integral taps are zero operands.
 *
 * A multiplier is described by an orc_mult: one of the two closed-form
 * kinds, or a table of 2^(2M) entries (carry << 23 | mantissa) that a user's
 * approx_mul produced through Algorithm 1 (Sec. V-A: the designer supplies
 * the C function; Sec. VI: LUTs are loaded at run time), plus the number E of
 * exponent bits of the simulated (1, E, M) format (Sec. V-B, last paragraph:
 * E from 1 to 8 given an exponent casting function).  Reading taken for the
 * casting function: an fp32 operand's exponent is re-biased to the E-bit
 * format's bias 2^(E-1) - 1 (IEEE convention: biased 0 is zero, all ones is
 * Inf/NaN); an operand below the format's smallest normal becomes a signed
 * zero and one above its largest binade a signed infinity; Algorithm 2 then
 * runs with that bias and that all-ones exponent, and the product's exponent
 * is re-biased back to fp32's.  E = 8 is fp32 itself (no change).
 *
 * Parity pins (tests/test_oracle_*.py): LUT byte sizes printed on the page;
 * exact kind == IEEE fp32 product of truncated operands; Mitchell hand values
 * and its log-domain definition; special-value invariants; brute force over
 * all mantissa pairs; GEMM/conv against numpy / torch-CPU float64 routines
 * on inputs where the exact kind is exact; user models through Algorithm 1
 * (a model computing the exact product gives the exact kind's table and
 * products bit for bit; an asymmetric model's hand-worked values); E-bit
 * formats (E = 5 against IEEE half ranges, hand-worked boundaries at E = 4,
 * the degenerate E = 1).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_EXACT 0
#define ORC_MITCHELL 1
#define ORC_TABLE 2

/* A simulated multiplier: closed-form kind or stored table, mantissa bits M
 * (1..11) and exponent bits E (1..8; 8 = fp32's own exponent). */
typedef struct {
    int kind;               /* ORC_EXACT, ORC_MITCHELL or ORC_TABLE */
    int M;
    int E;
    const uint32_t *table;  /* ORC_TABLE: entry of (p, q) at index p << M | q */
} orc_mult;

#define ORC_OK 0
#define ORC_EINVAL 1

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

static uint32_t sign_of(uint32_t x) { return x >> 31; }
static uint32_t bexp_of(uint32_t x) { return (x >> 23) & 0xFFu; }
static uint32_t frac_of(uint32_t x) { return x & 0x7FFFFFu; }

/* Top-M fraction bits of an fp32 pattern (truncation, no rounding). */
static uint32_t top_bits(uint32_t x, int M) { return frac_of(x) >> (23 - M); }

/*
 * The multiplier's functional model: the "user-defined C function approx_mul"
 * that Algorithm 1 is given.  Defined here for operands that are normal
 * numbers whose product is a normal number.  Both operands are first cut to
 * M fraction bits.  Mantissa values x, y in [0,1):
 *   exact    : (1+x)(1+y)
 *   mitchell : 1+x+y          if x+y < 1
 *              2(x+y)         otherwise
 * The result is scaled by 2^(ea+eb) (unbiased exponents) with the XOR sign.
 * All quantities are exact in double for M <= 11.
 */
float orc_approx_mul(int kind, int M, float a, float b)
{
    uint32_t ua = f2u(a), ub = f2u(b);
    double x = ldexp((double)top_bits(ua, M), -M);
    double y = ldexp((double)top_bits(ub, M), -M);
    double p;
    if (kind == ORC_EXACT) {
        p = (1.0 + x) * (1.0 + y);
    } else {
        p = (x + y < 1.0) ? (1.0 + x + y) : (2.0 * (x + y));
    }
    int e = (int)bexp_of(ua) - 127 + (int)bexp_of(ub) - 127;
    double c = ldexp(p, e);
    if (sign_of(ua) ^ sign_of(ub)) c = -c;
    return (float)c;
}

/* A multiplier model in Algorithm 1's terms: approx_mul(A, B) -> C. */
typedef float (*orc_model_fn)(const void *ctx, float A, float B);

typedef struct { int kind, M; } orc_kind_ctx;

static float kind_model(const void *ctx, float A, float B)
{
    const orc_kind_ctx *k = (const orc_kind_ctx *)ctx;
    return orc_approx_mul(k->kind, k->M, A, B);
}

/* A user's C function float approx_mul(float, float), as Sec. V-A has it. */
typedef float (*orc_user_fn)(float, float);
typedef struct { orc_user_fn fn; } orc_user_ctx;

static float user_model(const void *ctx, float A, float B)
{
    return ((const orc_user_ctx *)ctx)->fn(A, B);
}

/*
 * Algorithm 1 for one mantissa pair (p, q): build A = 1.p and B = 1.q with a
 * non-special exponent (biased 127 for both, so neither the operands nor the
 * product are special), call approx_mul, and detect the carry by comparing the
 * product's real biased exponent with the unnormalised one, eA + eB - 127.
 * Entry = carry << 23 | 23-bit mantissa of C.  Returns ORC_EINVAL when the
 * model's exponent moves by anything other than 0 or +1, or when the model
 * returns a negative product of two positive operands (the sign is Algorithm
 * 2's XOR, never the table's).
 */
static int algorithm1_entry(orc_model_fn approx_mul, const void *ctx, int M, uint32_t p, uint32_t q,
                            uint32_t *entry)
{
    if (M < 1 || M > 11) return ORC_EINVAL;
    if (p >= (1u << M) || q >= (1u << M)) return ORC_EINVAL;
    uint32_t ea = 127, eb = 127;
    float A = u2f((ea << 23) | (p << (23 - M)));
    float B = u2f((eb << 23) | (q << (23 - M)));
    float C = approx_mul(ctx, A, B);
    uint32_t uc = f2u(C);
    if (sign_of(uc)) return ORC_EINVAL;
    int un_normalized_exp = (int)ea + (int)eb - 127;
    int real_exp = (int)bexp_of(uc);
    int carry;
    if (real_exp == un_normalized_exp) carry = 0;
    else if (real_exp == un_normalized_exp + 1) carry = 1;
    else return ORC_EINVAL;
    *entry = ((uint32_t)carry << 23) | frac_of(uc);
    return ORC_OK;
}

/* All 2^(2M) entries of a model, row index p (first operand) high, q low. */
static int algorithm1_table(orc_model_fn approx_mul, const void *ctx, int M, uint32_t *out)
{
    if (M < 1 || M > 11) return ORC_EINVAL;
    uint32_t n = 1u << M;
    for (uint32_t p = 0; p < n; ++p)
        for (uint32_t q = 0; q < n; ++q) {
            int rc = algorithm1_entry(approx_mul, ctx, M, p, q, &out[(p << M) | q]);
            if (rc) return rc;
        }
    return ORC_OK;
}

int orc_lut_entry(int kind, int M, uint32_t p, uint32_t q, uint32_t *entry)
{
    if (kind != ORC_EXACT && kind != ORC_MITCHELL) return ORC_EINVAL;
    orc_kind_ctx k = {kind, M};
    return algorithm1_entry(kind_model, &k, M, p, q, entry);
}

int orc_lut(int kind, int M, uint32_t *out)
{
    if (kind != ORC_EXACT && kind != ORC_MITCHELL) return ORC_EINVAL;
    orc_kind_ctx k = {kind, M};
    return algorithm1_table(kind_model, &k, M, out);
}

/* Algorithm 1 over a user's approx_mul (the page's LUT-generation script). */
int orc_lut_from_fn(orc_user_fn approx_mul, int M, uint32_t *out)
{
    if (!approx_mul || !out) return ORC_EINVAL;
    orc_user_ctx u = {approx_mul};
    return algorithm1_table(user_model, &u, M, out);
}

static int mult_valid(const orc_mult *mu)
{
    if (!mu || mu->M < 1 || mu->M > 11 || mu->E < 1 || mu->E > 8) return 0;
    if (mu->kind == ORC_TABLE) return mu->table != NULL;
    return mu->kind == ORC_EXACT || mu->kind == ORC_MITCHELL;
}

/* The LUT entry of mantissa pair (qa, qb): read from the stored table, or
 * formed from the closed form through Algorithm 1. */
static int mult_entry(const orc_mult *mu, uint32_t qa, uint32_t qb, uint32_t *entry)
{
    if (mu->kind == ORC_TABLE) {
        *entry = mu->table[(qa << mu->M) | qb];
        return (*entry >> 24) ? ORC_EINVAL : ORC_OK;
    }
    return orc_lut_entry(mu->kind, mu->M, qa, qb, entry);
}

/* Operand classes after the exponent cast to the E-bit format. */
enum { CL_ZERO, CL_NORMAL, CL_INF, CL_NAN };

/*
 * The exponent casting function (reading stated in the header): fp32 operand
 * -> class and biased exponent of the (1, E, M) format with bias 2^(E-1) - 1.
 * Zero and denormal fp32 inputs are zero; fp32 Inf/NaN stay Inf/NaN; a normal
 * input whose re-biased exponent is not above zero is zero, one that reaches
 * the all-ones exponent 2^E - 1 is Inf.
 */
static int cast_operand(uint32_t x, int E, int *cexp)
{
    const int bias = (1 << (E - 1)) - 1;
    const int all_ones = (1 << E) - 1;
    uint32_t ex = bexp_of(x);
    if (ex == 255) return frac_of(x) ? CL_NAN : CL_INF;
    if (ex == 0) return CL_ZERO;
    int c = (int)ex - 127 + bias;
    if (c <= 0) return CL_ZERO;
    if (c >= all_ones) return CL_INF;
    *cexp = c;
    return CL_NORMAL;
}

/*
 * Algorithm 2 (AMSim) on fp32 bit patterns for a (1, E, M) multiplier:
 * sign XOR; index from the concatenated top-M mantissas; carry and mantissa
 * from the entry; e0 = eA + eB - bias; zero if e0 <= 0 or an input is zero;
 * Inf if e0 >= 2^E - 1; otherwise e = e0 + carry (Inf again if that reaches
 * 2^E - 1); the exponent is re-biased to fp32's for the result.
 */
static uint32_t algorithm2(const orc_mult *mu, uint32_t a, uint32_t b)
{
    const uint32_t QNAN = 0x7FC00000u;
    const int M = mu->M;
    const int bias = (1 << (mu->E - 1)) - 1;
    const int all_ones = (1 << mu->E) - 1;
    uint32_t s = sign_of(a) ^ sign_of(b);
    int ea = 0, eb = 0;
    int ca = cast_operand(a, mu->E, &ea), cb = cast_operand(b, mu->E, &eb);

    if (ca == CL_NAN || cb == CL_NAN) return QNAN;
    if (ca == CL_INF || cb == CL_INF) {
        if (ca == CL_ZERO || cb == CL_ZERO) return QNAN;
        return (s << 31) | 0x7F800000u;
    }
    if (ca == CL_ZERO || cb == CL_ZERO) return s << 31;

    /* Alg. 2: extract the top-M mantissas, concatenate into an index, fetch. */
    uint32_t qa = top_bits(a, M), qb = top_bits(b, M);
    uint32_t entry;
    if (mult_entry(mu, qa, qb, &entry) != ORC_OK) return QNAN;
    uint32_t carry = entry >> 23;
    uint32_t mant = entry & 0x7FFFFFu;

    int e0 = ea + eb - bias;
    if (e0 <= 0) return s << 31;                              /* underflow -> zero */
    if (e0 >= all_ones) return (s << 31) | 0x7F800000u;       /* overflow -> Inf  */
    int e = e0 + (int)carry;                                  /* normal case      */
    if (e >= all_ones) return (s << 31) | 0x7F800000u;
    return (s << 31) | ((uint32_t)(e - bias + 127) << 23) | mant;
}

/* AMSim for a closed-form kind with fp32's 8-bit exponent. */
uint32_t orc_amsim_bits(int kind, int M, uint32_t a, uint32_t b)
{
    orc_mult mu = {kind, M, 8, NULL};
    if (!mult_valid(&mu)) return 0x7FC00000u;
    return algorithm2(&mu, a, b);
}

uint32_t orc_amsim_mult_bits(const orc_mult *mu, uint32_t a, uint32_t b)
{
    if (!mult_valid(mu)) return 0x7FC00000u;
    return algorithm2(mu, a, b);
}

static float amsim(const orc_mult *mu, float a, float b)
{
    return u2f(algorithm2(mu, f2u(a), f2u(b)));
}

float orc_amsim(int kind, int M, float a, float b)
{
    return u2f(orc_amsim_bits(kind, M, f2u(a), f2u(b)));
}

int orc_mul(const orc_mult *mu, const float *a, const float *b, float *c, int64_t n)
{
    if (!mult_valid(mu)) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) c[i] = amsim(mu, a[i], b[i]);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* A small parallel-for over independent output items (no change of result). */

typedef void (*orc_item_fn)(void *ctx, int64_t item);
typedef struct { orc_item_fn fn; void *ctx; int64_t begin, end; } orc_span;

static void *orc_span_run(void *arg)
{
    orc_span *sp = (orc_span *)arg;
    for (int64_t i = sp->begin; i < sp->end; ++i) sp->fn(sp->ctx, i);
    return NULL;
}

static void orc_parallel(orc_item_fn fn, void *ctx, int64_t n, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        for (int64_t i = 0; i < n; ++i) fn(ctx, i);
        return;
    }
    pthread_t th[256];
    orc_span sp[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        sp[t].fn = fn; sp[t].ctx = ctx;
        sp[t].begin = n * t / nthreads; sp[t].end = n * (t + 1) / nthreads;
        if (pthread_create(&th[t], NULL, orc_span_run, &sp[t]) == 0) {
            ++started;
        } else {
            orc_span_run(&sp[t]);
            sp[t].fn = NULL;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (sp[t].fn) pthread_join(th[t], NULL);
    (void)started;
}

/* ------------------------------------------------------------------------ */
/* GEMM (row-major): C = alpha * op(A) op(B) + beta * C0, every product an
 * AMSim product of the multiplier `mu` with A's element as the first operand.  Only the listed rows
 * of C are produced: out[r*n + j] for r < nrows, plus sumabs = alpha-free
 * sum over k of |product|.  transA: A is stored k x m; transB: B is n x k.  */

typedef struct {
    orc_mult mu;
    int ta, tb, m, n, k;
    double alpha, beta;
    const float *A; int64_t lda;
    const float *B; int64_t ldb;
    const float *C0; int64_t ldc;
    const int *rows;
    float *out; double *sumabs;
} orc_gemm_ctx;

static void orc_gemm_row(void *vctx, int64_t r)
{
    orc_gemm_ctx *g = (orc_gemm_ctx *)vctx;
    int i = g->rows[r];
    for (int j = 0; j < g->n; ++j) {
        double s = 0.0, sa = 0.0;
        for (int kk = 0; kk < g->k; ++kk) {
            float a = g->ta ? g->A[(int64_t)kk * g->lda + i] : g->A[(int64_t)i * g->lda + kk];
            float b = g->tb ? g->B[(int64_t)j * g->ldb + kk] : g->B[(int64_t)kk * g->ldb + j];
            float p = amsim(&g->mu, a, b);
            s += (double)p;
            sa += fabs((double)p);
        }
        double v = g->alpha * s;
        if (g->beta != 0.0) v += g->beta * (double)g->C0[(int64_t)i * g->ldc + j];
        g->out[r * g->n + j] = (float)v;
        if (g->sumabs) g->sumabs[r * g->n + j] = sa;
    }
}

int orc_gemm_rows(const orc_mult *mu, int transA, int transB, int m, int n, int k,
                  double alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                  double beta, const float *C0, int64_t ldc,
                  const int *rows, int nrows, float *out, double *sumabs, int nthreads)
{
    if (!mult_valid(mu) || m < 0 || n < 0 || k < 0 || nrows < 0) return ORC_EINVAL;
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= m) return ORC_EINVAL;
    orc_gemm_ctx g = {*mu, transA, transB, m, n, k, alpha, beta,
                      A, lda, B, ldb, C0, ldc, rows, out, sumabs};
    orc_parallel(orc_gemm_row, &g, nrows, nthreads);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Conv2D, NHWC activations, RSCK (HWIO) filters, cross-correlation.
 * desc = {N,H,W,C,K,R,S, stride_h,stride_w, pad_h,pad_w, dil_h,dil_w}.
 * P = (H + 2 pad_h - dil_h (R-1) - 1) / stride_h + 1, likewise Q.
 * Out-of-range and non-integral taps are zero operands (IM2COL semantics). */

typedef struct {
    int N, H, W, C, K, R, S, sh, sw, ph, pw, dh, dw, P, Q;
} orc_conv;

static int orc_conv_init(const int *d, orc_conv *c)
{
    c->N = d[0]; c->H = d[1]; c->W = d[2]; c->C = d[3]; c->K = d[4]; c->R = d[5]; c->S = d[6];
    c->sh = d[7]; c->sw = d[8]; c->ph = d[9]; c->pw = d[10]; c->dh = d[11]; c->dw = d[12];
    if (c->N < 0 || c->H < 1 || c->W < 1 || c->C < 1 || c->K < 1 || c->R < 1 || c->S < 1) return ORC_EINVAL;
    if (c->sh < 1 || c->sw < 1 || c->ph < 0 || c->pw < 0 || c->dh < 1 || c->dw < 1) return ORC_EINVAL;
    int hh = c->H + 2 * c->ph - c->dh * (c->R - 1) - 1;
    int ww = c->W + 2 * c->pw - c->dw * (c->S - 1) - 1;
    if (hh < 0 || ww < 0) return ORC_EINVAL;
    c->P = hh / c->sh + 1;
    c->Q = ww / c->sw + 1;
    return ORC_OK;
}

typedef struct {
    orc_mult mu;
    orc_conv c;
    const float *x, *w, *dy;
    const int64_t *pts;
    float *out; double *sumabs;
} orc_conv_ctx;

static float x_at(const orc_conv *c, const float *x, int n, int h, int w, int ch)
{
    if (h < 0 || h >= c->H || w < 0 || w >= c->W) return 0.0f;
    return x[(((int64_t)n * c->H + h) * c->W + w) * c->C + ch];
}

/* Forward: Y[n,p,q,k] = sum_{r,s,c} X[n, p*sh - ph + r*dh, q*sw - pw + s*dw, c] * W[r,s,c,k]. */
static void orc_fwd_pt(void *vctx, int64_t t)
{
    orc_conv_ctx *g = (orc_conv_ctx *)vctx;
    const orc_conv *c = &g->c;
    int64_t idx = g->pts[t];
    int k = (int)(idx % c->K); idx /= c->K;
    int q = (int)(idx % c->Q); idx /= c->Q;
    int p = (int)(idx % c->P); idx /= c->P;
    int n = (int)idx;
    double s = 0.0, sa = 0.0;
    for (int r = 0; r < c->R; ++r)
        for (int ss = 0; ss < c->S; ++ss)
            for (int ch = 0; ch < c->C; ++ch) {
                float a = x_at(c, g->x, n, p * c->sh - c->ph + r * c->dh, q * c->sw - c->pw + ss * c->dw, ch);
                float b = g->w[(((int64_t)r * c->S + ss) * c->C + ch) * c->K + k];
                float pr = amsim(&g->mu, a, b);
                s += (double)pr; sa += fabs((double)pr);
            }
    g->out[t] = (float)s;
    if (g->sumabs) g->sumabs[t] = sa;
}

/* Preceding-layer gradient: dX[n,h,w,c] = sum_{r,s,k} dY[n,p,q,k] * W[r,s,c,k]
 * over p = (h + ph - r*dh)/sh, q = (w + pw - s*dw)/sw where integral and in range. */
static void orc_bwd_data_pt(void *vctx, int64_t t)
{
    orc_conv_ctx *g = (orc_conv_ctx *)vctx;
    const orc_conv *c = &g->c;
    int64_t idx = g->pts[t];
    int ch = (int)(idx % c->C); idx /= c->C;
    int w = (int)(idx % c->W); idx /= c->W;
    int h = (int)(idx % c->H); idx /= c->H;
    int n = (int)idx;
    double s = 0.0, sa = 0.0;
    for (int r = 0; r < c->R; ++r)
        for (int ss = 0; ss < c->S; ++ss)
            for (int k = 0; k < c->K; ++k) {
                int hp = h + c->ph - r * c->dh, wq = w + c->pw - ss * c->dw;
                float a = 0.0f;
                if (hp >= 0 && wq >= 0 && hp % c->sh == 0 && wq % c->sw == 0) {
                    int p = hp / c->sh, q = wq / c->sw;
                    if (p < c->P && q < c->Q)
                        a = g->dy[(((int64_t)n * c->P + p) * c->Q + q) * c->K + k];
                }
                float b = g->w[(((int64_t)r * c->S + ss) * c->C + ch) * c->K + k];
                float pr = amsim(&g->mu, a, b);
                s += (double)pr; sa += fabs((double)pr);
            }
    g->out[t] = (float)s;
    if (g->sumabs) g->sumabs[t] = sa;
}

/* Weight gradient: dW[r,s,c,k] = sum_{n,p,q} X[n, p*sh-ph+r*dh, q*sw-pw+s*dw, c] * dY[n,p,q,k]. */
static void orc_bwd_filter_pt(void *vctx, int64_t t)
{
    orc_conv_ctx *g = (orc_conv_ctx *)vctx;
    const orc_conv *c = &g->c;
    int64_t idx = g->pts[t];
    int k = (int)(idx % c->K); idx /= c->K;
    int ch = (int)(idx % c->C); idx /= c->C;
    int ss = (int)(idx % c->S); idx /= c->S;
    int r = (int)idx;
    double s = 0.0, sa = 0.0;
    for (int n = 0; n < c->N; ++n)
        for (int p = 0; p < c->P; ++p)
            for (int q = 0; q < c->Q; ++q) {
                float a = x_at(c, g->x, n, p * c->sh - c->ph + r * c->dh, q * c->sw - c->pw + ss * c->dw, ch);
                float b = g->dy[(((int64_t)n * c->P + p) * c->Q + q) * c->K + k];
                float pr = amsim(&g->mu, a, b);
                s += (double)pr; sa += fabs((double)pr);
            }
    g->out[t] = (float)s;
    if (g->sumabs) g->sumabs[t] = sa;
}

static int orc_conv_run(int which, const orc_mult *mu, const int *desc,
                        const float *x, const float *w, const float *dy,
                        const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    orc_conv_ctx g;
    if (!mult_valid(mu)) return ORC_EINVAL;
    if (orc_conv_init(desc, &g.c)) return ORC_EINVAL;
    int64_t total;
    if (which == 0) total = (int64_t)g.c.N * g.c.P * g.c.Q * g.c.K;
    else if (which == 1) total = (int64_t)g.c.N * g.c.H * g.c.W * g.c.C;
    else total = (int64_t)g.c.R * g.c.S * g.c.C * g.c.K;
    for (int64_t t = 0; t < npts; ++t)
        if (pts[t] < 0 || pts[t] >= total) return ORC_EINVAL;
    g.mu = *mu; g.x = x; g.w = w; g.dy = dy; g.pts = pts; g.out = out; g.sumabs = sumabs;
    orc_parallel(which == 0 ? orc_fwd_pt : which == 1 ? orc_bwd_data_pt : orc_bwd_filter_pt,
                 &g, npts, nthreads);
    return ORC_OK;
}

int orc_conv2d_fwd_points(const orc_mult *mu, const int *desc, const float *x, const float *w,
                          const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    return orc_conv_run(0, mu, desc, x, w, NULL, pts, npts, out, sumabs, nthreads);
}

int orc_conv2d_bwd_data_points(const orc_mult *mu, const int *desc, const float *dy, const float *w,
                               const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    return orc_conv_run(1, mu, desc, NULL, w, dy, pts, npts, out, sumabs, nthreads);
}

int orc_conv2d_bwd_filter_points(const orc_mult *mu, const int *desc, const float *x, const float *dy,
                                 const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    return orc_conv_run(2, mu, desc, x, NULL, dy, pts, npts, out, sumabs, nthreads);
}

int orc_conv2d_out_hw(const int *desc, int *P, int *Q)
{
    orc_conv c;
    if (orc_conv_init(desc, &c)) return ORC_EINVAL;
    *P = c.P; *Q = c.Q;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Depthwise Conv2D (Sec. III, Table I lists it beside Conv2D; it is the
 * convolution with one input channel per filter group).  Same descriptor,
 * K = C * D output channels for a channel multiplier D; the filter is
 * R x S x C x D and output channel k = c*D + d reads input channel c only:
 *   Y[n,p,q,c*D+d]  = sum_{r,s}   X[n, p*sh-ph+r*dh, q*sw-pw+s*dw, c] * W[r,s,c,d]
 *   dX[n,h,w,c]     = sum_{r,s,d} dY[n,p,q,c*D+d] * W[r,s,c,d]
 *                     over p = (h+ph-r*dh)/sh, q = (w+pw-s*dw)/sw integral, in range
 *   dW[r,s,c,d]     = sum_{n,p,q} X[n, p*sh-ph+r*dh, q*sw-pw+s*dw, c] * dY[n,p,q,c*D+d]
 * Operand order as for Conv2D: (x, w), (dy, w), (x, dy). */

static void orc_dw_fwd_pt(void *vctx, int64_t t)
{
    orc_conv_ctx *g = (orc_conv_ctx *)vctx;
    const orc_conv *c = &g->c;
    const int D = c->K / c->C;
    int64_t idx = g->pts[t];
    int k = (int)(idx % c->K); idx /= c->K;
    int q = (int)(idx % c->Q); idx /= c->Q;
    int p = (int)(idx % c->P); idx /= c->P;
    int n = (int)idx;
    int ch = k / D, d = k % D;
    double s = 0.0, sa = 0.0;
    for (int r = 0; r < c->R; ++r)
        for (int ss = 0; ss < c->S; ++ss) {
            float a = x_at(c, g->x, n, p * c->sh - c->ph + r * c->dh, q * c->sw - c->pw + ss * c->dw, ch);
            float b = g->w[(((int64_t)r * c->S + ss) * c->C + ch) * D + d];
            float pr = amsim(&g->mu, a, b);
            s += (double)pr; sa += fabs((double)pr);
        }
    g->out[t] = (float)s;
    if (g->sumabs) g->sumabs[t] = sa;
}

static void orc_dw_bwd_data_pt(void *vctx, int64_t t)
{
    orc_conv_ctx *g = (orc_conv_ctx *)vctx;
    const orc_conv *c = &g->c;
    const int D = c->K / c->C;
    int64_t idx = g->pts[t];
    int ch = (int)(idx % c->C); idx /= c->C;
    int w = (int)(idx % c->W); idx /= c->W;
    int h = (int)(idx % c->H); idx /= c->H;
    int n = (int)idx;
    double s = 0.0, sa = 0.0;
    for (int r = 0; r < c->R; ++r)
        for (int ss = 0; ss < c->S; ++ss)
            for (int d = 0; d < D; ++d) {
                int hp = h + c->ph - r * c->dh, wq = w + c->pw - ss * c->dw;
                float a = 0.0f;
                if (hp >= 0 && wq >= 0 && hp % c->sh == 0 && wq % c->sw == 0) {
                    int p = hp / c->sh, q = wq / c->sw;
                    if (p < c->P && q < c->Q)
                        a = g->dy[(((int64_t)n * c->P + p) * c->Q + q) * c->K + ch * D + d];
                }
                float b = g->w[(((int64_t)r * c->S + ss) * c->C + ch) * D + d];
                float pr = amsim(&g->mu, a, b);
                s += (double)pr; sa += fabs((double)pr);
            }
    g->out[t] = (float)s;
    if (g->sumabs) g->sumabs[t] = sa;
}

static void orc_dw_bwd_filter_pt(void *vctx, int64_t t)
{
    orc_conv_ctx *g = (orc_conv_ctx *)vctx;
    const orc_conv *c = &g->c;
    const int D = c->K / c->C;
    int64_t idx = g->pts[t];
    int d = (int)(idx % D); idx /= D;
    int ch = (int)(idx % c->C); idx /= c->C;
    int ss = (int)(idx % c->S); idx /= c->S;
    int r = (int)idx;
    double s = 0.0, sa = 0.0;
    for (int n = 0; n < c->N; ++n)
        for (int p = 0; p < c->P; ++p)
            for (int q = 0; q < c->Q; ++q) {
                float a = x_at(c, g->x, n, p * c->sh - c->ph + r * c->dh, q * c->sw - c->pw + ss * c->dw, ch);
                float b = g->dy[(((int64_t)n * c->P + p) * c->Q + q) * c->K + ch * D + d];
                float pr = amsim(&g->mu, a, b);
                s += (double)pr; sa += fabs((double)pr);
            }
    g->out[t] = (float)s;
    if (g->sumabs) g->sumabs[t] = sa;
}

static int orc_dw_run(int which, const orc_mult *mu, const int *desc,
                      const float *x, const float *w, const float *dy,
                      const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    orc_conv_ctx g;
    if (!mult_valid(mu)) return ORC_EINVAL;
    if (orc_conv_init(desc, &g.c)) return ORC_EINVAL;
    if (g.c.K % g.c.C) return ORC_EINVAL;
    int64_t total;
    if (which == 0) total = (int64_t)g.c.N * g.c.P * g.c.Q * g.c.K;
    else if (which == 1) total = (int64_t)g.c.N * g.c.H * g.c.W * g.c.C;
    else total = (int64_t)g.c.R * g.c.S * g.c.K;
    for (int64_t t = 0; t < npts; ++t)
        if (pts[t] < 0 || pts[t] >= total) return ORC_EINVAL;
    g.mu = *mu; g.x = x; g.w = w; g.dy = dy; g.pts = pts; g.out = out; g.sumabs = sumabs;
    orc_parallel(which == 0 ? orc_dw_fwd_pt : which == 1 ? orc_dw_bwd_data_pt : orc_dw_bwd_filter_pt,
                 &g, npts, nthreads);
    return ORC_OK;
}

int orc_dwconv2d_fwd_points(const orc_mult *mu, const int *desc, const float *x, const float *w,
                            const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    return orc_dw_run(0, mu, desc, x, w, NULL, pts, npts, out, sumabs, nthreads);
}

int orc_dwconv2d_bwd_data_points(const orc_mult *mu, const int *desc, const float *dy, const float *w,
                                 const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    return orc_dw_run(1, mu, desc, NULL, w, dy, pts, npts, out, sumabs, nthreads);
}

int orc_dwconv2d_bwd_filter_points(const orc_mult *mu, const int *desc, const float *x, const float *dy,
                                   const int64_t *pts, int64_t npts, float *out, double *sumabs, int nthreads)
{
    return orc_dw_run(2, mu, desc, x, NULL, dy, pts, npts, out, sumabs, nthreads);
}
