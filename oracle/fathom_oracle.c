/*
 * fathom_oracle.c -- plain, slow CPU oracle for the Fathom variable-depth
 * bit-plane key scan.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke
 * check and the benchmark's CPU-baseline leg are the only callers.  The
 * product path (the CUDA library) never links, loads or calls this file, and
 * this file includes no header of the product path.
 *
 * Source: the review page "Fathom: 쿼리마다 깊이를 바꾸는 스캔으로 1M 토큰
 * 디코딩을 1.67배 빠르게 하다" (jaehun.me, a summary of the Fathom paper).
 * Sections cited below are the paper's, as the page cites them:
 *   §2   evaluation protocol (first 4 / last 32 tokens kept, top k-36 rest)
 *   §3.2 bit-plane K cache (quantiser, planes, prefix dequantisation)
 *   §3.3 per-query read depth (g_j, reverse water-filling, 30-step bisection)
 *   §3.5 KLT-rotated basis
 *   §3.4 per-layer budgets (flat, greedy)
 *   §3.6 host-resident store as contiguous runs, fixed-size run list
 *   §4/§5 fidelity: relative L2 error against dense and exact top-k attention
 *   Appx. A toy example (6 keys x 4 channels, 2 query heads)
 *
 * Arithmetic: fp64 for everything the pages leave open; the plan's decisions
 * (depths, theta) use only IEEE-exact operations (mul, add, sqrt, compare) in
 * a fixed order so that any IEEE implementation reproduces them bit for bit.
 * Compile with -O2 -ffp-contract=off (no FMA contraction, no fast-math).
 *
 * Readings of points the pages leave open (each is listed in the design notes):
 *   R1 the stored block scale is a rounded to fp16 (round-to-nearest-even,
 *      saturating at 65504); that same fp16 value is used to code and to
 *      dequantise, so the prefix identity holds for the stored scale.
 *   R2 floor(k/s) is the floor of the exact real quotient.
 *   R3 a16 == 0 makes every code 8 (value 0).
 *   R4 token i of a block is bit i of the plane word (bit 0 = first token).
 *   R5 tail tokens (i >= n in the last block) have all-zero bits, take no part
 *      in the block maximum and are never scored or selected.
 *   R6 g_j = (sum_h q_hj^2) * Var_j, h ascending, fp64.
 *   R7 depth t_j(theta) = #{m in 0..3 : g_j >= theta * 2^(2m+1)}, which is
 *      clip(round-half-up(log4(g_j/theta)), 0, 4).
 *   R8 auto bracket: hi = max g (all depths 0), lo = min_{g>0} g / 512 (all
 *      positive-g channels at depth 4); when depth(lo) fits the budget the
 *      bisection is skipped and theta = lo.
 *   R9 selection ties: lower token index wins; output ascending by index.
 *   R10 attention scale 1/sqrt(D); no mass redistribution.
 *   R21 the greedy per-layer plan starts every layer at the lowest budget and
 *      adds one budget step at a time to the layer whose measured error falls
 *      the most, until the budgets average the target.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PLANES 4

/* ------------------------------------------------------------------------ */
/* fp16 / bf16 helpers (R1)                                                  */
/* ------------------------------------------------------------------------ */

/* Round a non-negative finite float to the nearest fp16 value (ties to even),
 * saturating at the largest finite fp16 value 65504.  Returns the value. */
double oracle_round_fp16(double a)
{
    if (a <= 0.0) return 0.0;
    if (a >= 65504.0) return 65504.0;
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) */
    /* fp16 normal numbers carry 11 significant bits; below 2^-14 the step is
     * fixed at 2^-24 (subnormals). */
    double quantum = (e - 1 >= -14) ? ldexp(1.0, e - 11) : ldexp(1.0, -24);
    double r = rint(a / quantum); /* default rounding mode: ties to even */
    double v = r * quantum;
    if (v > 65504.0) v = 65504.0;
    return v;
}

/* Encode a non-negative fp16-representable value as its 16-bit pattern. */
uint16_t oracle_fp16_bits(double v)
{
    if (v == 0.0) return 0;
    if (v < ldexp(1.0, -14)) return (uint16_t)(v / ldexp(1.0, -24));
    int e;
    double m = frexp(v, &e);      /* v = m * 2^e, m in [0.5, 1) */
    int biased = e - 1 + 15;
    int mant = (int)((m * 2.0 - 1.0) * 1024.0);
    return (uint16_t)((biased << 10) | mant);
}

double oracle_fp16_value(uint16_t h)
{
    int exp = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double sgn = (h & 0x8000) ? -1.0 : 1.0;
    if (exp == 0) return sgn * ldexp((double)mant, -24);
    return sgn * ldexp(1024.0 + mant, exp - 25);
}

double oracle_bf16_value(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* §3.2  4-bit symmetric per-channel quantiser over 64-token blocks          */
/* ------------------------------------------------------------------------ */

/* Code of one value:  c = clip(floor(k/s), -8, 7) + 8  with s = a16/8.
 * floor is the floor of the exact quotient (R2): the fp64 quotient is
 * corrected with exact products, which are exact because |f| <= 16 here and
 * s carries 11 significant bits. */
int oracle_code(float k, double a16)
{
    if (a16 == 0.0) return 8;                       /* R3 */
    double s = a16 / 8.0;                           /* exact */
    double kk = (double)k;
    double q = kk / s;
    if (q >= 16.0) return 15;
    if (q <= -16.0) return 0;
    double f = floor(q);
    if (f * s > kk) f -= 1.0;                       /* exact checks */
    if ((f + 1.0) * s <= kk) f += 1.0;
    if (f < -8.0) f = -8.0;
    if (f > 7.0) f = 7.0;
    return (int)f + 8;
}

/* Quantise and pack one store.
 *   keys   [U][n][D] fp32 (row-major: token, channel)
 *   planes [U][D][4][nb] u64, plane p = 0 is the MSB of the code (§3.2);
 *          bit i of a word is token 64*beta + i (R4).
 *   scales [U][D][nb] fp16 bits of a16 (R1).
 *   codes  optional [U][n][D] u8 (the 4-bit codes), NULL to skip.
 * nb = ceil(n/64).  Returns 0. */
int oracle_quantize_pack(int U, int n, int D, const float *keys,
                         uint64_t *planes, uint16_t *scales, uint8_t *codes)
{
    int nb = (n + 63) / 64;
    for (int u = 0; u < U; ++u) {
        const float *K = keys + (size_t)u * n * D;
        for (int j = 0; j < D; ++j) {
            for (int beta = 0; beta < nb; ++beta) {
                int i0 = beta * 64;
                int i1 = i0 + 64 < n ? i0 + 64 : n;
                /* a_{beta,j} = max_{i in beta} |k_ij| */
                double a = 0.0;
                for (int i = i0; i < i1; ++i) {
                    double v = fabs((double)K[(size_t)i * D + j]);
                    if (v > a) a = v;
                }
                double a16 = oracle_round_fp16(a);
                scales[((size_t)u * D + j) * nb + beta] = oracle_fp16_bits(a16);
                uint64_t P[ORACLE_PLANES] = {0, 0, 0, 0};
                for (int i = i0; i < i1; ++i) {
                    int c = oracle_code(K[(size_t)i * D + j], a16);
                    if (codes) codes[((size_t)u * n + i) * D + j] = (uint8_t)c;
                    for (int p = 0; p < ORACLE_PLANES; ++p) {
                        uint64_t bit = (uint64_t)((c >> (3 - p)) & 1);
                        P[p] |= bit << (i - i0);
                    }
                }
                for (int p = 0; p < ORACLE_PLANES; ++p)
                    planes[(((size_t)u * D + j) * ORACLE_PLANES + p) * nb + beta] = P[p];
            }
        }
    }
    return 0;
}

/* Prefix dequantisation (§3.2): reading the first t planes gives
 * c_t = c >> (4 - t) and the value (c_t + 0.5 - 2^(t-1)) * a / 2^(t-1).
 * t = 0 contributes nothing. */
double oracle_dequant(int c_t, int t, double a16)
{
    if (t <= 0) return 0.0;
    double half = ldexp(1.0, t - 1);
    return ((double)c_t + 0.5 - half) * a16 / half;
}

/* Read the first t planes of token i, channel j of unit u from a store laid
 * out [U][D][4][nb]: the code prefix c_t. */
static int read_prefix(const uint64_t *planes, int D, int nb, int u, int j, int i, int t)
{
    int beta = i / 64, bit = i % 64;
    int c_t = 0;
    for (int p = 0; p < t; ++p) {
        uint64_t w = planes[(((size_t)u * D + j) * ORACLE_PLANES + p) * nb + beta];
        c_t = (c_t << 1) | (int)((w >> bit) & 1u);
    }
    return c_t;
}

/* ------------------------------------------------------------------------ */
/* §3.3  channel importance and reverse water-filling                       */
/* ------------------------------------------------------------------------ */

/* g_j = (sum_h q_hj^2) * Var_j   (R6).  q [G][D] fp32, var [D] fp32. */
void oracle_importance(int D, int G, const float *q, const float *var, double *g)
{
    for (int j = 0; j < D; ++j) {
        double s = 0.0;
        for (int h = 0; h < G; ++h) {
            double x = (double)q[(size_t)h * D + j];
            s = s + x * x;
        }
        g[j] = s * (double)var[j];
    }
}

/* t_j(theta) = #{m in 0..3 : g_j >= theta * 2^(2m+1)}   (R7) */
int oracle_depth_of(double g, double theta)
{
    int t = 0;
    for (int m = 0; m < 4; ++m)
        if (g >= theta * ldexp(1.0, 2 * m + 1)) ++t;
    return t;
}

static int total_depth(int D, const double *g, double theta)
{
    int s = 0;
    for (int j = 0; j < D; ++j) s += oracle_depth_of(g[j], theta);
    return s;
}

/* Reverse water-filling: minimise sum_j g_j 4^-t_j subject to sum_j t_j <= B
 * with t_j = clip(round(log4(g_j/theta)), 0, 4); theta is found by 30 steps
 * of log (geometric-mean) bisection and is the smallest tried theta that fits
 * the budget (§3.3, Appx. A).
 *   bracket  NULL for the automatic bracket (R8), else {lo, hi}.
 *   trace    optional [30] probes and trace_sum [30] their total depths
 *            (entries past the last step are left untouched).
 * Writes depth[D] and *theta; returns the number of bisection steps run. */
int oracle_plan(int D, int G, const float *q, const float *var, int B,
                const double *bracket, uint8_t *depth, double *theta,
                double *trace, int *trace_sum)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)D);
    oracle_importance(D, G, q, var, g);
    double lo, hi;
    int steps = 0;
    if (bracket) {
        lo = bracket[0];
        hi = bracket[1];
    } else {
        double gmax = 0.0, gmin = 0.0;
        for (int j = 0; j < D; ++j) {
            if (g[j] > gmax) gmax = g[j];
            if (g[j] > 0.0 && (gmin == 0.0 || g[j] < gmin)) gmin = g[j];
        }
        if (gmax == 0.0) {                 /* nothing to read */
            for (int j = 0; j < D; ++j) depth[j] = 0;
            *theta = 0.0;
            free(g);
            return 0;
        }
        hi = gmax;
        lo = gmin / 512.0;
        if (total_depth(D, g, lo) <= B) {  /* budget not binding */
            for (int j = 0; j < D; ++j) depth[j] = (uint8_t)oracle_depth_of(g[j], lo);
            *theta = lo;
            free(g);
            return 0;
        }
    }
    for (int it = 0; it < 30; ++it) {
        double mid = sqrt(lo * hi);
        int s = total_depth(D, g, mid);
        if (trace) trace[it] = mid;
        if (trace_sum) trace_sum[it] = s;
        if (s <= B) hi = mid; else lo = mid;
        ++steps;
    }
    for (int j = 0; j < D; ++j) depth[j] = (uint8_t)oracle_depth_of(g[j], hi);
    *theta = hi;
    free(g);
    return steps;
}

/* Fixed-depth comparison plan (the byte-equivalent of a 136-bit scan): the
 * n_sel channels of largest g_j (ties: lower j) at depth t_fixed, others 0. */
void oracle_plan_fixed(int D, int G, const float *q, const float *var,
                       int n_sel, int t_fixed, uint8_t *depth)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)D);
    oracle_importance(D, G, q, var, g);
    for (int j = 0; j < D; ++j) {
        int better = 0;   /* channels ranked ahead of j */
        for (int i = 0; i < D; ++i)
            if (g[i] > g[j] || (g[i] == g[j] && i < j)) ++better;
        depth[j] = (uint8_t)(better < n_sel ? t_fixed : 0);
    }
    free(g);
}

/* §3.6  fixed-size run list: one slot per channel, zero length when
 * inactive.  Offsets are in 64-bit words / fp16 scales, relative to the
 * unit's store (src) and the unit's staging area (dst), channels ascending.
 * runs[D][6] = {src_word, n_words, dst_word, src_scale, n_scales, dst_scale} */
void oracle_runs(int D, int n, const uint8_t *depth, uint32_t *runs)
{
    uint32_t nb = (uint32_t)((n + 63) / 64);
    uint32_t dst_w = 0, dst_s = 0;
    for (int j = 0; j < D; ++j) {
        uint32_t t = depth[j];
        uint32_t *r = runs + (size_t)j * 6;
        r[0] = (uint32_t)j * ORACLE_PLANES * nb;
        r[1] = t * nb;
        r[2] = dst_w;
        r[3] = (uint32_t)j * nb;
        r[4] = t > 0 ? nb : 0;
        r[5] = dst_s;
        dst_w += r[1];
        dst_s += r[4];
    }
}

/* §3.6 gather: copy each active channel's run and its scales from the store
 * into the staging area.  store_planes/scales are one unit's store, stage_*
 * one unit's staging area. */
void oracle_gather(int D, const uint32_t *runs, const uint64_t *store_planes,
                   const uint16_t *store_scales, uint64_t *stage_planes,
                   uint16_t *stage_scales)
{
    for (int j = 0; j < D; ++j) {
        const uint32_t *r = runs + (size_t)j * 6;
        for (uint32_t w = 0; w < r[1]; ++w) stage_planes[r[2] + w] = store_planes[r[0] + w];
        for (uint32_t s = 0; s < r[4]; ++s) stage_scales[r[5] + s] = store_scales[r[3] + s];
    }
}

/* ------------------------------------------------------------------------ */
/* §3.2/§3.3/§7  approximate scores                                          */
/* ------------------------------------------------------------------------ */

/* s_h(i) = sum_{j : t_j > 0} q_hj * khat_ij, khat from the first t_j planes.
 * planes/scales [U][D][4][nb] / [U][D][nb]; depth [U][D]; q [U][G][D];
 * scores [U][G][n] fp64. */
void oracle_scores(int U, int n, int D, int G, const uint64_t *planes,
                   const uint16_t *scales, const uint8_t *depth, const float *q,
                   double *scores)
{
    int nb = (n + 63) / 64;
    for (int u = 0; u < U; ++u)
        for (int h = 0; h < G; ++h)
            for (int i = 0; i < n; ++i) {
                double s = 0.0;
                for (int j = 0; j < D; ++j) {
                    int t = depth[(size_t)u * D + j];
                    if (t == 0) continue;
                    int c_t = read_prefix(planes, D, nb, u, j, i, t);
                    double a16 = oracle_fp16_value(scales[((size_t)u * D + j) * nb + i / 64]);
                    s += (double)q[((size_t)u * G + h) * D + j] * oracle_dequant(c_t, t, a16);
                }
                scores[((size_t)u * G + h) * n + i] = s;
            }
}

/* Same as oracle_scores, but reading the staging layout produced by the run
 * list (channels' first t_j planes at dst_word, scales at dst_scale).  Used to
 * check that a staged scan reads what the in-place scan reads. */
void oracle_scores_staged(int n, int D, int G, const uint32_t *runs,
                          const uint64_t *stage_planes, const uint16_t *stage_scales,
                          const uint8_t *depth, const float *q, double *scores)
{
    int nb = (n + 63) / 64;
    for (int h = 0; h < G; ++h)
        for (int i = 0; i < n; ++i) {
            double s = 0.0;
            for (int j = 0; j < D; ++j) {
                int t = depth[j];
                if (t == 0) continue;
                const uint32_t *r = runs + (size_t)j * 6;
                int c_t = 0;
                for (int p = 0; p < t; ++p) {
                    uint64_t w = stage_planes[r[2] + (uint32_t)p * nb + (uint32_t)(i / 64)];
                    c_t = (c_t << 1) | (int)((w >> (i % 64)) & 1u);
                }
                double a16 = oracle_fp16_value(stage_scales[r[5] + (uint32_t)(i / 64)]);
                s += (double)q[(size_t)h * D + j] * oracle_dequant(c_t, t, a16);
            }
            scores[(size_t)h * n + i] = s;
        }
}

/* ------------------------------------------------------------------------ */
/* §2  selection: forced sink/recent tokens plus top (k - |forced|)          */
/* ------------------------------------------------------------------------ */

typedef struct { double s; int i; } cand_t;

static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->s > b->s) return -1;          /* score descending */
    if (a->s < b->s) return 1;
    return (a->i < b->i) ? -1 : (a->i > b->i);   /* R9 */
}

static int int_cmp(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

/* scores [G][n] (one unit); idx/sel_scores [G][k].  The forced set is the
 * first min(n_sink, n) and the last min(n_recent, n) tokens.  Requires
 * |forced| <= k <= n; returns -1 otherwise, 0 on success. */
int oracle_select(int n, int G, const double *scores, int k, int n_sink,
                  int n_recent, int32_t *idx, double *sel_scores)
{
    if (k > n) return -1;
    char *forced = (char *)calloc((size_t)n, 1);
    int nf = 0;
    for (int i = 0; i < n; ++i)
        if (i < n_sink || i >= n - n_recent) { forced[i] = 1; ++nf; }
    if (nf > k) { free(forced); return -1; }
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
    int *out = (int *)malloc(sizeof(int) * (size_t)(k > 0 ? k : 1));
    for (int h = 0; h < G; ++h) {
        const double *s = scores + (size_t)h * n;
        int m = 0, o = 0;
        for (int i = 0; i < n; ++i) {
            if (forced[i]) out[o++] = i;
            else { c[m].s = s[i]; c[m].i = i; ++m; }
        }
        qsort(c, (size_t)m, sizeof(cand_t), cand_cmp);
        for (int r = 0; r < k - nf; ++r) out[o++] = c[r].i;
        qsort(out, (size_t)k, sizeof(int), int_cmp);
        for (int r = 0; r < k; ++r) {
            idx[(size_t)h * k + r] = out[r];
            if (sel_scores) sel_scores[(size_t)h * k + r] = s[out[r]];
        }
    }
    free(c); free(out); free(forced);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* §1/§2  exact attention over each head's selected rows                    */
/* ------------------------------------------------------------------------ */

/* o_h = sum_{i in S_h} softmax_i(q_h . k_i / sqrt(D)) v_i over bf16 rows
 * widened exactly, fp64 throughout (R10).
 *   krows/vrows [n][D] bf16 bits; q [G][D]; idx [G][k]; out [G][D]. */
void oracle_attention(int n, int D, int G, const uint16_t *krows,
                      const uint16_t *vrows, const float *q, const int32_t *idx,
                      int k, double *out)
{
    (void)n;
    double *logit = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    double scale = 1.0 / sqrt((double)D);
    for (int h = 0; h < G; ++h) {
        double mx = -INFINITY;
        for (int r = 0; r < k; ++r) {
            int i = idx[(size_t)h * k + r];
            double d = 0.0;
            for (int j = 0; j < D; ++j)
                d += (double)q[(size_t)h * D + j] * oracle_bf16_value(krows[(size_t)i * D + j]);
            logit[r] = d * scale;
            if (logit[r] > mx) mx = logit[r];
        }
        double den = 0.0;
        for (int j = 0; j < D; ++j) out[(size_t)h * D + j] = 0.0;
        for (int r = 0; r < k; ++r) {
            double p = exp(logit[r] - mx);
            den += p;
            int i = idx[(size_t)h * k + r];
            for (int j = 0; j < D; ++j)
                out[(size_t)h * D + j] += p * oracle_bf16_value(vrows[(size_t)i * D + j]);
        }
        for (int j = 0; j < D; ++j) out[(size_t)h * D + j] /= den;
    }
    free(logit);
}

/* ------------------------------------------------------------------------ */
/* §4/§5 fidelity references and §3.4 greedy per-layer budgets               */
/* ------------------------------------------------------------------------ */

/* §7 (the store as the K cache): every token's key rebuilt from all four
 * planes of its block and channel, k_ij = dequant(c_ij, 4, a_{i/64, j}).
 *   planes [D][4][cb], scales [D][cb] of one unit; keys [n][D] (out). */
void oracle_reconstruct(int n, int D, int cb, const uint64_t *planes, const uint16_t *scales,
                        double *keys)
{
    for (int i = 0; i < n; ++i) {
        int beta = i / 64, bit = i % 64;
        for (int j = 0; j < D; ++j) {
            int c = 0;
            for (int p = 0; p < ORACLE_PLANES; ++p) {
                uint64_t w = planes[((size_t)j * ORACLE_PLANES + p) * cb + beta];
                c = (c << 1) | (int)((w >> bit) & 1u);
            }
            keys[(size_t)i * D + j] = oracle_dequant(c, 4, oracle_fp16_value(scales[(size_t)j * cb + beta]));
        }
    }
}

/* Attention as oracle_attention with the keys given as fp64 values
 * keys [n][D] (the rebuilt keys), values still bf16 rows. */
void oracle_attention_keys(int n, int D, int G, const double *keys, const uint16_t *vrows,
                           const float *q, const int32_t *idx, int k, double *out)
{
    (void)n;
    double *logit = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    double scale = 1.0 / sqrt((double)D);
    for (int h = 0; h < G; ++h) {
        double mx = -INFINITY;
        for (int r = 0; r < k; ++r) {
            int i = idx[(size_t)h * k + r];
            double d = 0.0;
            for (int j = 0; j < D; ++j)
                d += (double)q[(size_t)h * D + j] * keys[(size_t)i * D + j];
            logit[r] = d * scale;
            if (logit[r] > mx) mx = logit[r];
        }
        double den = 0.0;
        for (int j = 0; j < D; ++j) out[(size_t)h * D + j] = 0.0;
        for (int r = 0; r < k; ++r) {
            double p = exp(logit[r] - mx);
            den += p;
            int i = idx[(size_t)h * k + r];
            for (int j = 0; j < D; ++j)
                out[(size_t)h * D + j] += p * oracle_bf16_value(vrows[(size_t)i * D + j]);
        }
        for (int j = 0; j < D; ++j) out[(size_t)h * D + j] /= den;
    }
    free(logit);
}

/* Exact score of every token, the quantity the exact top-k ranks:
 * s_h(i) = sum_j q_hj k_ij over the key rows widened exactly, fp64.
 *   keys [n][D] fp32, q [G][D] fp32, out [G][n]. */
void oracle_exact_scores(int n, int D, int G, const float *keys, const float *q, double *out)
{
    for (int h = 0; h < G; ++h)
        for (int i = 0; i < n; ++i) {
            double d = 0.0;
            for (int j = 0; j < D; ++j)
                d += (double)q[(size_t)h * D + j] * (double)keys[(size_t)i * D + j];
            out[(size_t)h * n + i] = d;
        }
}

/* Greedy per-layer plan (§3.4, reading R21): budget levels b_min + step*i,
 * i = 0 .. levels-1; err [layers][levels].  Every layer starts at level 0;
 * layers*(b_mean-b_min)/step times, one level is added to the layer whose
 * error drops the most on its next level (the lowest such layer on a tie),
 * skipping layers already at the top level.  budgets [layers] (out). */
void oracle_greedy_budgets(int layers, int levels, const double *err, int b_min, int step,
                           int b_mean, int32_t *budgets)
{
    int *lev = (int *)calloc((size_t)layers, sizeof(int));
    int incs = layers * (b_mean - b_min) / step;
    for (int it = 0; it < incs; ++it) {
        int best = -1;
        double best_drop = 0.0;
        for (int l = 0; l < layers; ++l) {
            if (lev[l] == levels - 1) continue;
            double drop = err[l * levels + lev[l]] - err[l * levels + lev[l] + 1];
            if (best == -1 || drop > best_drop) { best = l; best_drop = drop; }
        }
        if (best == -1) break;
        lev[best] += 1;
    }
    for (int l = 0; l < layers; ++l) budgets[l] = b_min + step * lev[l];
    free(lev);
}

/* ------------------------------------------------------------------------ */
/* §3.3 calibration statistics and §3.5 KLT basis                            */
/* ------------------------------------------------------------------------ */

/* Per-channel mean and unbiased (ddof = 1) variance of calibration keys
 * keys [m][D]; cov optional [D][D] unbiased covariance. */
void oracle_calibrate(int m, int D, const float *keys, double *mean, double *var,
                      double *cov)
{
    for (int j = 0; j < D; ++j) {
        double s = 0.0;
        for (int i = 0; i < m; ++i) s += (double)keys[(size_t)i * D + j];
        mean[j] = s / (double)m;
    }
    for (int j = 0; j < D; ++j) {
        double s = 0.0;
        for (int i = 0; i < m; ++i) {
            double d = (double)keys[(size_t)i * D + j] - mean[j];
            s += d * d;
        }
        var[j] = s / (double)(m - 1);
    }
    if (cov) {
        for (int a = 0; a < D; ++a)
            for (int b = 0; b < D; ++b) {
                double s = 0.0;
                for (int i = 0; i < m; ++i)
                    s += ((double)keys[(size_t)i * D + a] - mean[a]) *
                         ((double)keys[(size_t)i * D + b] - mean[b]);
                cov[(size_t)a * D + b] = s / (double)(m - 1);
            }
    }
}

/* Eigen-decomposition of a symmetric D x D matrix by cyclic Jacobi rotations
 * (fp64).  On return lam[D] holds the eigenvalues in descending order and
 * V[D][D] the matching eigenvectors as columns (V[j][c] = component j of
 * eigenvector c), each scaled so that its largest-magnitude component is
 * positive.  Returns the number of sweeps. */
int oracle_eigh(int D, const double *A_in, double *lam, double *V)
{
    double *A = (double *)malloc(sizeof(double) * (size_t)D * D);
    memcpy(A, A_in, sizeof(double) * (size_t)D * D);
    for (int a = 0; a < D; ++a)
        for (int b = 0; b < D; ++b) V[(size_t)a * D + b] = (a == b) ? 1.0 : 0.0;
    int sweep;
    for (sweep = 0; sweep < 100; ++sweep) {
        double off = 0.0, tot = 0.0;
        for (int a = 0; a < D; ++a)
            for (int b = 0; b < D; ++b) {
                double x = A[(size_t)a * D + b] * A[(size_t)a * D + b];
                tot += x;
                if (a != b) off += x;
            }
        if (off <= 1e-30 * tot || off == 0.0) break;
        for (int p = 0; p < D - 1; ++p)
            for (int r = p + 1; r < D; ++r) {
                double apr = A[(size_t)p * D + r];
                if (apr == 0.0) continue;
                double app = A[(size_t)p * D + p], arr = A[(size_t)r * D + r];
                /* rotation angle that zeroes A[p][r] */
                double tau = (arr - app) / (2.0 * apr);
                double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                double c = 1.0 / sqrt(1.0 + t * t), s = t * c;
                for (int x = 0; x < D; ++x) {   /* columns p, r */
                    double axp = A[(size_t)x * D + p], axr = A[(size_t)x * D + r];
                    A[(size_t)x * D + p] = c * axp - s * axr;
                    A[(size_t)x * D + r] = s * axp + c * axr;
                }
                for (int x = 0; x < D; ++x) {   /* rows p, r */
                    double apx = A[(size_t)p * D + x], arx = A[(size_t)r * D + x];
                    A[(size_t)p * D + x] = c * apx - s * arx;
                    A[(size_t)r * D + x] = s * apx + c * arx;
                }
                for (int x = 0; x < D; ++x) {   /* accumulate V = V * J */
                    double vxp = V[(size_t)x * D + p], vxr = V[(size_t)x * D + r];
                    V[(size_t)x * D + p] = c * vxp - s * vxr;
                    V[(size_t)x * D + r] = s * vxp + c * vxr;
                }
            }
    }
    for (int a = 0; a < D; ++a) lam[a] = A[(size_t)a * D + a];
    /* selection sort by eigenvalue, descending */
    for (int a = 0; a < D; ++a) {
        int best = a;
        for (int b = a + 1; b < D; ++b) if (lam[b] > lam[best]) best = b;
        if (best != a) {
            double tl = lam[a]; lam[a] = lam[best]; lam[best] = tl;
            for (int x = 0; x < D; ++x) {
                double tv = V[(size_t)x * D + a];
                V[(size_t)x * D + a] = V[(size_t)x * D + best];
                V[(size_t)x * D + best] = tv;
            }
        }
    }
    for (int c = 0; c < D; ++c) {       /* sign: largest |component| positive */
        int arg = 0;
        for (int x = 1; x < D; ++x)
            if (fabs(V[(size_t)x * D + c]) > fabs(V[(size_t)arg * D + c])) arg = x;
        if (V[(size_t)arg * D + c] < 0.0)
            for (int x = 0; x < D; ++x) V[(size_t)x * D + c] = -V[(size_t)x * D + c];
    }
    free(A);
    return sweep;
}

/* §3.5 rotated keys k' = (k - mu) V, fp64 accumulate, written as fp32.
 * keys [n][D] fp32, mu [D], V [D][D] (columns = basis vectors). */
void oracle_rotate(int n, int D, const float *keys, const double *mu,
                   const double *V, float *out)
{
    for (int i = 0; i < n; ++i)
        for (int c = 0; c < D; ++c) {
            double s = 0.0;
            for (int j = 0; j < D; ++j)
                s += ((double)keys[(size_t)i * D + j] - mu[j]) * V[(size_t)j * D + c];
            out[(size_t)i * D + c] = (float)s;
        }
}

/* §3.5 rotated queries q' = q V (fp64). q [G][D] fp32, out [G][D] fp64. */
void oracle_rotate_query(int G, int D, const float *q, const double *V, double *out)
{
    for (int h = 0; h < G; ++h)
        for (int c = 0; c < D; ++c) {
            double s = 0.0;
            for (int j = 0; j < D; ++j) s += (double)q[(size_t)h * D + j] * V[(size_t)j * D + c];
            out[(size_t)h * D + c] = s;
        }
}
