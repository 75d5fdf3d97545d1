/*
 * moe_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * route / dispatch / combine path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path never does.
 * It shares no source, header, table or helper with the CUDA library, and it
 * owns its own bf16 and e4m3 codecs, written from the format definitions.
 *
 * Sources (page title, section):
 *   [PMC] "Efficient and portable mixture-of-experts communication"
 *         (Perplexity blog, 2025-04-02; read in its Indonesian translation
 *         "Komunikasi mixture-of-experts yang efisien dan portabel").
 *   [DBO] "Dual Batch Overlap" (vLLM design documentation).
 *
 * Readings taken where the pages are silent (each pinned by the CPU tests):
 *   - Top-k selects on the fp32 logits, largest first; equal logits go to the
 *     lower expert index (-0.0 and +0.0 are equal).
 *   - Routing weights are the softmax renormalised over the k selected
 *     experts, evaluated in double, then rounded to float.
 *   - Within one expert, rows are filled in ascending token order. A pair
 *     whose position reaches the capacity C is dropped (slot -1), counted,
 *     and contributes nothing to combine (no renormalisation).
 *   - fp8 dispatch: per 128-element block, scale = amax/448 in fp32 (1 when
 *     amax is 0), q = e4m3(x / scale) with round-to-nearest-even and
 *     saturation to +-448.
 *   - Combine accumulates in fp32 with one fused multiply-add per selected
 *     expert, in selection order, from 0, then rounds to bf16 (nearest-even).
 *   - The grouped GEMM that stands in for the experts maps each dispatched
 *     fp8 row through one random e4m3 weight matrix per expert (128 x 128
 *     weight blocks with an fp32 scale each), exactly, then rounds once to
 *     bf16 (nearest-even); each dispatched bf16 row through one random bf16
 *     weight matrix per expert, in double, then once to bf16.
 *
 * Layouts (row-major):
 *   logits[T][E] f32; topk_idx[T][k] i32; topk_w[T][k] f32; slot[T][k] i32;
 *   x[T][H] bf16 bits; recv_x[E][C][H] bf16 bits or recv_q[E][C][H] e4m3 codes;
 *   recv_scale[E][C][H/128] f32; recv_src[E][C] i32; y[E][C][H] bf16 bits;
 *   out[T][H] bf16 bits. Expert e lives on virtual rank e / (E/R); its rows are
 *   [e*C, (e+1)*C), so [R][E/R][C][H] and [E][C][H] are the same memory.
 *
 * Every function returns 0 on success and -1 on an invalid argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 (1 sign, 8 exponent, 7 fraction bits): the upper half of an IEEE-754 */
/* binary32. Decoding appends 16 zero bits. Encoding keeps the upper 16 bits */
/* and rounds on the discarded lower 16 bits: above half -> up, below -> down, */
/* exactly half -> to the even upper value. NaN stays NaN (quiet bit set).    */
/* ------------------------------------------------------------------------ */
static float bf16_decode(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint16_t bf16_encode_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;             /* a carry into the exponent is the correct result */
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------------ */
/* OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign, 4 exponent bits    */
/* with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN.           */
/*   exponent field 0:      value = (m/8) * 2^(1-7)            (subnormal)   */
/*   exponent field 1..15:  value = (1 + m/8) * 2^(e-7)                      */
/* Largest finite magnitude: S.1111.110 = 1.75 * 2^8 = 448.                  */
/* ------------------------------------------------------------------------ */
static double e4m3_magnitude(unsigned code7)      /* code without the sign bit */
{
    unsigned e = (code7 >> 3) & 15u, m = code7 & 7u;
    if (e == 0)
        return ldexp((double)m / 8.0, 1 - 7);
    return ldexp(1.0 + (double)m / 8.0, (int)e - 7);
}

static float e4m3_decode(uint8_t code)
{
    if ((code & 0x7Fu) == 0x7Fu)
        return NAN;
    double v = e4m3_magnitude(code & 0x7Fu);
    return (float)((code & 0x80u) ? -v : v);
}

/* The 127 finite non-negative magnitudes, ascending with the code (0..126). */
static double g_e4m3_mag[127];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void)
{
    if (g_e4m3_ready)
        return;
    for (unsigned c = 0; c < 127; ++c)
        g_e4m3_mag[c] = e4m3_magnitude(c);
    g_e4m3_ready = 1;
}

/* Nearest finite E4M3 value, ties to the even code, magnitudes above 448
 * saturate to 448 (the "satfinite" reading). NaN maps to the NaN code. */
static uint8_t e4m3_encode_rne_satfinite(float f)
{
    if (isnan(f))
        return 0x7Fu;
    uint8_t sign = signbit(f) ? 0x80u : 0x00u;
    double a = fabs((double)f);
    if (a >= g_e4m3_mag[126])
        return (uint8_t)(sign | 126u);
    /* binary search: the largest code lo with magnitude <= a */
    unsigned lo = 0, hi = 126;             /* mag[lo] <= a < mag[hi] */
    while (hi - lo > 1) {
        unsigned mid = (lo + hi) / 2;
        if (g_e4m3_mag[mid] <= a)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = a - g_e4m3_mag[lo], dhi = g_e4m3_mag[hi] - a;
    unsigned c;
    if (dlo < dhi)
        c = lo;
    else if (dhi < dlo)
        c = hi;
    else
        c = (lo & 1u) ? hi : lo;           /* tie: the even code */
    return (uint8_t)(sign | c);
}

/* ------------------------------------------------------------------------ */
/* Codec entry points (used by the tests that pin the codecs).               */
/* ------------------------------------------------------------------------ */
void oracle_bf16_encode(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_encode_rne(in[i]);
}

void oracle_bf16_decode(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_decode(in[i]);
}

void oracle_e4m3_encode(const float *in, uint8_t *out, int64_t n)
{
    e4m3_table_init();
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_encode_rne_satfinite(in[i]);
}

void oracle_e4m3_decode(const uint8_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_decode(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Step 1: router top-k and routing weights.                                 */
/* [PMC §Introduction]: the router yields a probability distribution over    */
/* the experts, the experts with the top-K scores are chosen, and each       */
/* token's output is a weighted average whose weights come from that         */
/* distribution. The distribution is a softmax of the logits; restricted to  */
/* the k chosen experts and renormalised it is                               */
/*     w_j = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0),                       */
/* where l_0 is the largest logit (same value as the full softmax's          */
/* probabilities divided by their sum over the chosen set).                  */
/* ------------------------------------------------------------------------ */
typedef struct {
    float l;
    int32_t e;
} scored_expert;

static int by_logit_desc_then_index(const void *pa, const void *pb)
{
    const scored_expert *a = (const scored_expert *)pa, *b = (const scored_expert *)pb;
    if (a->l > b->l) return -1;
    if (a->l < b->l) return 1;
    return (a->e < b->e) ? -1 : (a->e > b->e) ? 1 : 0;   /* equal logits: lower index first */
}

int oracle_route(int32_t T, int32_t E, int32_t k, const float *logits,
                 int32_t *topk_idx, float *topk_w, double *topk_w64 /* may be NULL */)
{
    if (T < 0 || E < 1 || k < 1 || k > E)
        return -1;
    scored_expert *row = (scored_expert *)malloc(sizeof(scored_expert) * (size_t)E);
    double *ex = (double *)malloc(sizeof(double) * (size_t)k);
    if (!row || !ex) {
        free(row);
        free(ex);
        return -1;
    }
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) {
            row[e].l = logits[(int64_t)t * E + e];
            row[e].e = e;
        }
        qsort(row, (size_t)E, sizeof(scored_expert), by_logit_desc_then_index);
        double top = (double)row[0].l, sum = 0.0;
        for (int32_t j = 0; j < k; ++j) {
            ex[j] = exp((double)row[j].l - top);
            sum += ex[j];
        }
        for (int32_t j = 0; j < k; ++j) {
            double w = ex[j] / sum;
            topk_idx[(int64_t)t * k + j] = row[j].e;
            topk_w[(int64_t)t * k + j] = (float)w;
            if (topk_w64)
                topk_w64[(int64_t)t * k + j] = w;
        }
    }
    free(row);
    free(ex);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: per-expert histogram, exclusive scan, slot of every (t, j).       */
/* [PMC §Dispatch]: a counting warp tallies how many tokens go to each       */
/* destination expert. [PMC §Portable kernels]: the maximum number of tokens */
/* is fixed, which bounds what one expert receives and lets every sender     */
/* compute a unique destination address without synchronising. Here that     */
/* bound is the capacity C and the address of pair (t, j) is row             */
/* e*C + slot[t][j], the slot being the number of earlier tokens that chose  */
/* the same expert. offsets[] is the exclusive scan of the raw counts        */
/* (E+1 entries); rank_counts[r] counts the rows that land on virtual rank r.*/
/* ------------------------------------------------------------------------ */
int oracle_count(int32_t T, int32_t E, int32_t k, int32_t R, int32_t C,
                 const int32_t *topk_idx, int32_t *counts, int32_t *offsets,
                 int32_t *slot, int32_t *rank_counts, int32_t *dropped)
{
    if (T < 0 || E < 1 || k < 1 || k > E || R < 1 || E % R != 0 || C < 1)
        return -1;
    int32_t *cursor = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!cursor)
        return -1;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = topk_idx[(int64_t)t * k + j];
            if (e < 0 || e >= E) {
                free(cursor);
                return -1;
            }
            int32_t pos = cursor[e]++;
            slot[(int64_t)t * k + j] = (pos < C) ? pos : -1;
        }
    }
    int32_t run = 0, lost = 0, per_rank = E / R;
    for (int32_t r = 0; r < R; ++r)
        rank_counts[r] = 0;
    for (int32_t e = 0; e < E; ++e) {
        counts[e] = cursor[e];
        offsets[e] = run;
        run += cursor[e];
        rank_counts[e / per_rank] += (cursor[e] < C) ? cursor[e] : C;
        lost += (cursor[e] > C) ? cursor[e] - C : 0;
    }
    offsets[E] = run;
    *dropped = lost;
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: dispatch. [PMC §Dispatch]: the tokens are unpacked into one        */
/* tensor for the grouped expert GEMM, all tokens of one expert grouped      */
/* together whatever their source, and the token's origin is stored beside   */
/* it so that combine knows where each row goes back to.                     */
/* bf16: a bit copy of the row to every kept slot; recv_src holds the token. */
/* ------------------------------------------------------------------------ */
int oracle_dispatch_bf16(int32_t T, int32_t H, int32_t E, int32_t k, int32_t C,
                         const uint16_t *x, const int32_t *topk_idx, const int32_t *slot,
                         uint16_t *recv_x, int32_t *recv_src)
{
    if (T < 0 || H < 1 || E < 1 || k < 1 || C < 1)
        return -1;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = topk_idx[(int64_t)t * k + j], s = slot[(int64_t)t * k + j];
            if (s < 0)
                continue;
            int64_t row = (int64_t)e * C + s;
            memcpy(recv_x + row * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);
            recv_src[row] = t;
        }
    }
    return 0;
}

/* fp8: [PMC §Dispatch] sends the tokens together with their block scaling   */
/* factors. One fp32 scale per 128 elements: scale = amax/448 (1 when the    */
/* block is all zero), q = e4m3(x/scale) with fp32 division. The token is    */
/* quantised once and the same codes and scales go to every kept slot.       */
int oracle_dispatch_fp8(int32_t T, int32_t H, int32_t E, int32_t k, int32_t C,
                        const uint16_t *x, const int32_t *topk_idx, const int32_t *slot,
                        uint8_t *recv_q, float *recv_scale, int32_t *recv_src)
{
    if (T < 0 || H < 128 || H % 128 != 0 || E < 1 || k < 1 || C < 1)
        return -1;
    e4m3_table_init();
    const int32_t nb = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *sc = (float *)malloc(sizeof(float) * (size_t)nb);
    if (!q || !sc) {
        free(q);
        free(sc);
        return -1;
    }
    for (int32_t t = 0; t < T; ++t) {
        const uint16_t *xr = x + (int64_t)t * H;
        for (int32_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int32_t i = 0; i < 128; ++i) {
                float a = fabsf(bf16_decode(xr[b * 128 + i]));
                if (a > amax)
                    amax = a;
            }
            float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
            sc[b] = scale;
            for (int32_t i = 0; i < 128; ++i)
                q[b * 128 + i] = e4m3_encode_rne_satfinite(bf16_decode(xr[b * 128 + i]) / scale);
        }
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = topk_idx[(int64_t)t * k + j], s = slot[(int64_t)t * k + j];
            if (s < 0)
                continue;
            int64_t row = (int64_t)e * C + s;
            memcpy(recv_q + row * H, q, (size_t)H);
            memcpy(recv_scale + row * nb, sc, sizeof(float) * (size_t)nb);
            recv_src[row] = t;
        }
    }
    free(q);
    free(sc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Source-rank offsets inside each expert. [PMC §Dispatch]: the receiver     */
/* groups all tokens of one expert together across the data-parallel ranks  */
/* that sent them. Token t comes from source rank t / tps (tps tokens per    */
/* rank; tps = 0: one rank), S = max(1, ceil(T / tps)). For s = 0 .. S:      */
/*   src_offsets[e][s] = number of kept pairs (t, j) with topk_idx = e and   */
/*                       source rank of t below s,                           */
/* counted over the pairs, so it does not depend on where dispatch put them. */
/* ------------------------------------------------------------------------ */
int oracle_src_offsets(int32_t T, int32_t E, int32_t k, int32_t tps, const int32_t *topk_idx,
                       const int32_t *slot, int32_t *src_offsets)
{
    if (T < 0 || E < 1 || k < 1 || tps < 0)
        return -1;
    const int32_t per = tps > 0 ? tps : (T > 0 ? T : 1);
    const int32_t S = T > 0 ? (int32_t)(((int64_t)T + per - 1) / per) : 1;
    memset(src_offsets, 0, sizeof(int32_t) * (size_t)E * (size_t)(S + 1));
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            if (slot[(int64_t)t * k + j] < 0)
                continue;
            const int32_t e = topk_idx[(int64_t)t * k + j];
            src_offsets[(int64_t)e * (S + 1) + t / per + 1] += 1;    /* counted at every s above t's rank */
        }
    }
    for (int32_t e = 0; e < E; ++e)
        for (int32_t s = 1; s <= S; ++s)
            src_offsets[(int64_t)e * (S + 1) + s] += src_offsets[(int64_t)e * (S + 1) + s - 1];
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Synthetic expert (stands in for the grouped GEMM of [PMC §Dispatch]):     */
/*   bf16 input:  y = bf16(float(x) * s_e)                                   */
/*   fp8 input:   y = bf16((float(q) * scale) * s_e)                         */
/* on the first min(counts[e], C) rows of every expert; other rows untouched.*/
/* ------------------------------------------------------------------------ */
int oracle_expert_synthetic(int32_t H, int32_t E, int32_t C, int32_t fp8,
                            const void *recv, const float *recv_scale,
                            const int32_t *counts, const float *s, uint16_t *y)
{
    if (H < 1 || E < 1 || C < 1 || (fp8 && H % 128 != 0))
        return -1;
    const int32_t nb = H / 128;
    for (int32_t e = 0; e < E; ++e) {
        int32_t rows = counts[e] < C ? counts[e] : C;
        for (int32_t r = 0; r < rows; ++r) {
            int64_t row = (int64_t)e * C + r;
            for (int32_t h = 0; h < H; ++h) {
                float v;
                if (fp8) {
                    float deq = e4m3_decode(((const uint8_t *)recv)[row * H + h]) * recv_scale[row * nb + h / 128];
                    v = deq * s[e];
                } else {
                    v = bf16_decode(((const uint16_t *)recv)[row * H + h]) * s[e];
                }
                y[row * H + h] = bf16_encode_rne(v);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped expert GEMM on the fp8 dispatch layout (stands in for the experts  */
/* that consume the dispatched, block-scaled tokens of [PMC §Dispatch];      */
/* random weights, one linear map of N outputs per expert, no activation):   */
/*   y[e][r][n] = bf16( sum_b  a_scale[e][r][b] * w_scale[e][n/128][b]        */
/*                      * sum_{i in block b} q[e][r][i] * w[e][n][i] )        */
/* q: the dispatched e4m3 codes, a_scale: their scale per 128 inputs;        */
/* w[e][N][K]: e4m3 weight codes, w_scale[e][N/128][K/128]: one scale per    */
/* 128 x 128 weight block. Each inner block sum is exact in double (an e4m3  */
/* product has at most 8 significant bits, between 2^-18 and 2^18, and 128   */
/* of them need fewer than 53 bits); the outer sum is taken in double and    */
/* the result rounded once to bf16, to nearest, ties to even. The sums      */
/* start from +0, so an exact zero comes out as +0.                          */
/* ------------------------------------------------------------------------ */

/* Nearest bf16 to a double, ties to the even code; beyond the largest      */
/* finite bf16 (plus half an ulp) the result is infinite.                   */
static uint16_t bf16_encode_rne_double(double v)
{
    if (isnan(v))
        return 0x7FC0u;
    const uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);                        /* a = m * 2^ex, m in [0.5, 1)   */
    int q = ex - 8;                       /* 8 significant bits: grid 2^q  */
    if (q < -133)
        q = -133;                         /* bf16 subnormal grid           */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);   /* ties to even (default mode) */
    if (r > 3.3895313892515355e38)        /* largest finite bf16            */
        return sign | 0x7F80u;
    float f = (float)r;                   /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFFu);
}

/* One output row: y_row[n] for n < N from one dispatched row (K inputs). */
int oracle_gemm_fp8_row(int32_t K, int32_t N, const uint8_t *q_row, const float *a_scale_row,
                        const uint8_t *w, const float *w_scale, uint16_t *y_row)
{
    if (K < 128 || N < 128 || K % 128 != 0 || N % 128 != 0)
        return -1;
    const int32_t kb = K / 128;
    for (int32_t n = 0; n < N; ++n) {
        const uint8_t *wn = w + (int64_t)n * K;
        double acc = 0.0;
        for (int32_t b = 0; b < kb; ++b) {
            double block = 0.0;
            for (int32_t i = b * 128; i < (b + 1) * 128; ++i)
                block += (double)e4m3_decode(q_row[i]) * (double)e4m3_decode(wn[i]);
            acc += (double)a_scale_row[b] * (double)w_scale[(int64_t)(n / 128) * kb + b] * block;
        }
        y_row[n] = bf16_encode_rne_double(acc);
    }
    return 0;
}

/* Every expert, rows r < min(counts[e], C); other rows untouched.
 * recv_q[E][C][K], recv_scale[E][C][K/128], w[E][N][K],
 * w_scale[E][N/128][K/128], y[E][C][N]. */
int oracle_expert_gemm_fp8(int32_t K, int32_t N, int32_t E, int32_t C, const uint8_t *recv_q,
                           const float *recv_scale, const int32_t *counts, const uint8_t *w,
                           const float *w_scale, uint16_t *y)
{
    if (E < 1 || C < 1 || K < 128 || N < 128 || K % 128 != 0 || N % 128 != 0)
        return -1;
    const int32_t kb = K / 128;
    for (int32_t e = 0; e < E; ++e) {
        const int32_t rows = counts[e] < C ? counts[e] : C;
        const uint8_t *we = w + (int64_t)e * N * K;
        const float *se = w_scale + (int64_t)e * (N / 128) * kb;
        for (int32_t r = 0; r < rows; ++r) {
            const int64_t row = (int64_t)e * C + r;
            if (oracle_gemm_fp8_row(K, N, recv_q + row * K, recv_scale + row * kb, we, se, y + row * N) != 0)
                return -1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Grouped expert GEMM on the bf16 dispatch layout (the same stand-in for the */
/* experts, for bf16 rows; random bf16 weights, one map of N outputs each):   */
/*   y[e][r][n] = bf16( sum_i x[e][r][i] * w[e][n][i] )                       */
/* The products and the sum are taken in double (a bf16 product has at most  */
/* 16 significant bits; the sum rounds only far below bf16 precision) and    */
/* the result is rounded once to bf16, to nearest, ties to even; an exact    */
/* zero comes out as +0.                                                     */
/* ------------------------------------------------------------------------ */
int oracle_gemm_bf16_row(int32_t K, int32_t N, const uint16_t *x_row, const uint16_t *w, uint16_t *y_row)
{
    if (K < 1 || N < 1)
        return -1;
    for (int32_t n = 0; n < N; ++n) {
        const uint16_t *wn = w + (int64_t)n * K;
        double acc = 0.0;
        for (int32_t i = 0; i < K; ++i)
            acc += (double)bf16_decode(x_row[i]) * (double)bf16_decode(wn[i]);
        y_row[n] = bf16_encode_rne_double(acc);
    }
    return 0;
}

/* Every expert, rows r < min(counts[e], C); other rows untouched.
 * recv_x[E][C][K] bf16, w[E][N][K] bf16, y[E][C][N] bf16. */
int oracle_expert_gemm_bf16(int32_t K, int32_t N, int32_t E, int32_t C, const uint16_t *recv_x,
                            const int32_t *counts, const uint16_t *w, uint16_t *y)
{
    if (E < 1 || C < 1 || K < 1 || N < 1)
        return -1;
    for (int32_t e = 0; e < E; ++e) {
        const int32_t kept_rows = counts[e] < C ? counts[e] : C;
        const uint16_t *we = w + (int64_t)e * N * K;
        for (int32_t r = 0; r < kept_rows; ++r) {
            const int64_t row = (int64_t)e * C + r;
            if (oracle_gemm_bf16_row(K, N, recv_x + row * K, we, y + row * N) != 0)
                return -1;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 4: combine. [PMC §Combine]: the receiver reads every expert's        */
/* 16-bit output row through the routing table and forms the weighted sum    */
/* with the router's weights, writing an externally allocated tensor:        */
/*   out[t] = bf16( sum_j w[t][j] * y[e_j][slot_j] ),                        */
/* accumulated in fp32 with one fused multiply-add per j in selection order, */
/* starting from zero; dropped pairs (slot -1) are skipped.                  */
/* ------------------------------------------------------------------------ */
int oracle_combine(int32_t T, int32_t H, int32_t E, int32_t k, int32_t C,
                   const uint16_t *y, const int32_t *topk_idx, const float *topk_w,
                   const int32_t *slot, uint16_t *out)
{
    if (T < 0 || H < 1 || E < 1 || k < 1 || C < 1)
        return -1;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t j = 0; j < k; ++j) {
                int32_t s = slot[(int64_t)t * k + j];
                if (s < 0)
                    continue;
                int64_t row = (int64_t)topk_idx[(int64_t)t * k + j] * C + s;
                acc = fmaf(topk_w[(int64_t)t * k + j], bf16_decode(y[row * H + h]), acc);
            }
            out[(int64_t)t * H + h] = bf16_encode_rne(acc);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Stand-in for the layer compute around the MoE block in the dual-batch-    */
/* overlap schedule ([DBO §Introduction]: A0 = qkv projection, A1 = core      */
/* attention + out projection + MoE gate, S = shared expert):                */
/*   out[i] = bf16(float(in[i]) * a)   (fp32 product, round to nearest even). */
/* ------------------------------------------------------------------------ */
int oracle_scale_rows(int64_t n, const uint16_t *in, float a, uint16_t *out)
{
    if (n < 0)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_encode_rne(bf16_decode(in[i]) * a);
    return 0;
}
