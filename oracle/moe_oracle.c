/*
 * moe_oracle.c -- plain, slow CPU oracle of the routed-experts MoE step over
 * NVFP4 expert weights.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *
 *   y_t = sum_{j=0..k-1, valid} w_tj * W_down[e_tj] ( SiLU(W_gate[e_tj] x_t) (.) (W_up[e_tj] x_t) )
 *
 * the routed-experts step the serving pages build their "lna2" kernel for
 * ("LNA-CANON.md", section "lna2 とは": resident expert teams, rows per expert
 * R_e, m <= 24; "dsv4-carve" README, section "house kernel lna2").  The pages'
 * EXL3 trellis format is never defined there, so the expert weights are NVFP4
 * (the format the V100 page, section 7.1, adopts because it expands into FP16
 * in registers): an E2M1 value times its 16-element block's E4M3 scale times
 * the (expert, projection) FP32 tensor scale.
 *
 * Precision: every dequantised weight is formed exactly in double
 * (E2M1 x E4M3 x fp32 needs at most 2+4+24 significant bits); x (bf16) and the
 * routing weights (fp32) convert to double exactly; dot products, SiLU and the
 * combine run in double, each sum in plain index order.  The result is the
 * definition's value up to double rounding.
 *
 * Slot rules (the pages are silent; plainest reading): an id < 0 is an empty
 * slot and contributes nothing; an id >= E contributes nothing and is counted
 * as bad; duplicate ids within a token are independent slots.
 *
 * Grouping (the pairs-by-expert tables an expert-team kernel works from):
 * counts[e] = number of valid pairs with id e; offsets = exclusive prefix sum
 * (offsets[E] = number of valid pairs); perm lists the flat pair indices
 * p = t*k + j of valid pairs sorted by (expert, p) -- a stable counting sort,
 * the unique answer.
 *
 * Routing (the step in front of the path, which the pages do not describe):
 * per token the k largest router logits in descending order, equal logits by
 * the smaller expert index, NaN as -infinity, and the softmax of the selected
 * logits in double -- the plain definition of top-k gating.
 *
 * Parallelism: optional OpenMP over independent output rows only; every
 * individual sum keeps its sequential order, so the result does not depend on
 * the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- formats */

/* E2M1 (OCP Microscaling formats v1.0, FP4 E2M1): bit 3 sign, bits 2..1
 * exponent with bias 1, bit 0 mantissa; exponent 0 is subnormal (0 or 0.5). */
double oracle_dec_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* E4M3FN (OCP 8-bit floating point, E4M3): bit 7 sign, bits 6..3 exponent
 * with bias 7, bits 2..0 mantissa; exponent 0 is subnormal (m/8 * 2^-6);
 * S.1111.111 is NaN; there is no infinity (max 448). */
double oracle_dec_e4m3(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15u && m == 7u)
        return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* Value tables built from the two definitions above (code -> value). */
static double tab_e2m1[16], tab_e4m3[256];
static int tabs_ready = 0;

static void build_tables(void)
{
    if (tabs_ready)
        return;
    for (unsigned c = 0; c < 16; ++c)
        tab_e2m1[c] = oracle_dec_e2m1(c);
    for (unsigned c = 0; c < 256; ++c)
        tab_e4m3[c] = oracle_dec_e4m3(c);
    tabs_ready = 1;
}

/* bf16 bit pattern -> double (exact). */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One dequantised weight: row r, column c of a [rows, K] NVFP4 matrix whose
 * packed bytes start at q (K/2 bytes per row) and scales at s (K/16 per row). */
static double weight_at(const uint8_t *q, const uint8_t *s, double ts, int K, size_t r, int c)
{
    uint8_t byte = q[r * (size_t)(K / 2) + (size_t)(c / 2)];
    unsigned nib = (c & 1) ? (byte >> 4) : (byte & 15u);
    uint8_t sc = s[r * (size_t)(K / 16) + (size_t)(c / 16)];
    return tab_e2m1[nib] * tab_e4m3[sc] * ts;
}

/* Dequantise a whole [rows, K] matrix into out (double, row-major). */
void oracle_dequant(const uint8_t *q, const uint8_t *s, float ts, int rows, int K, double *out)
{
    build_tables();
    for (size_t r = 0; r < (size_t)rows; ++r)
        for (int c = 0; c < K; ++c)
            out[r * (size_t)K + (size_t)c] = weight_at(q, s, (double)ts, K, r, c);
}

static int n_threads_eff(int n)
{
#ifdef _OPENMP
    return n > 0 ? n : omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* ---------------------------------------------------------------- one pair */

/* One (token, expert) pair: xr (double [H]) through expert e.
 *   g[i] = sum_c Wg[e][i][c] x[c]      u[i] likewise       (i < I)
 *   h[i] = g[i] / (1 + exp(-g[i])) * u[i]
 *   o[r] = sum_i Wd[e][r][i] h[i]      (r < H)
 * Any of g, u, h may be NULL (scratch is then allocated internally). */
static void quant_row_nvfp4(const float *v, int n, double *out);

/* The pair, with h quantised once to NVFP4 before the down projection when
 * act != 0 (rounded to fp32, then quant_row_nvfp4). */
static void expert_pair_q(int H, int I, int e, const double *xr,
                          const uint8_t *gate_q, const uint8_t *gate_s, const float *gate_ts,
                          const uint8_t *up_q, const uint8_t *up_s, const float *up_ts,
                          const uint8_t *down_q, const uint8_t *down_s, const float *down_ts,
                          double *g, double *u, double *h, double *o, int n_threads, int act)
{
    build_tables();
    double *gbuf = g ? g : (double *)malloc(sizeof(double) * (size_t)I);
    double *ubuf = u ? u : (double *)malloc(sizeof(double) * (size_t)I);
    double *hbuf = h ? h : (double *)malloc(sizeof(double) * (size_t)I);
    const uint8_t *gq = gate_q + (size_t)e * I * (H / 2), *gs = gate_s + (size_t)e * I * (H / 16);
    const uint8_t *uq = up_q + (size_t)e * I * (H / 2), *us = up_s + (size_t)e * I * (H / 16);
    const uint8_t *dq = down_q + (size_t)e * H * (I / 2), *ds = down_s + (size_t)e * H * (I / 16);
    double tg = (double)gate_ts[e], tu = (double)up_ts[e], td = (double)down_ts[e];
    int nt = n_threads_eff(n_threads);
    (void)nt;

#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int i = 0; i < I; ++i) {
        double sg = 0.0, su = 0.0;
        for (int c = 0; c < H; ++c) {
            sg += weight_at(gq, gs, tg, H, (size_t)i, c) * xr[c];
            su += weight_at(uq, us, tu, H, (size_t)i, c) * xr[c];
        }
        gbuf[i] = sg;
        ubuf[i] = su;
        hbuf[i] = sg / (1.0 + exp(-sg)) * su;
    }
    if (act) {
        float *hf = (float *)malloc(sizeof(float) * (size_t)I);
        for (int i = 0; i < I; ++i)
            hf[i] = (float)hbuf[i];
        quant_row_nvfp4(hf, I, hbuf);
        free(hf);
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int r = 0; r < H; ++r) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += weight_at(dq, ds, td, I, (size_t)r, i) * hbuf[i];
        o[r] = acc;
    }
    if (!g) free(gbuf);
    if (!u) free(ubuf);
    if (!h) free(hbuf);
}

void oracle_expert_pair(int H, int I, int e, const double *xr,
                        const uint8_t *gate_q, const uint8_t *gate_s, const float *gate_ts,
                        const uint8_t *up_q, const uint8_t *up_s, const float *up_ts,
                        const uint8_t *down_q, const uint8_t *down_s, const float *down_ts,
                        double *g, double *u, double *h, double *o, int n_threads)
{
    expert_pair_q(H, I, e, xr, gate_q, gate_s, gate_ts, up_q, up_s, up_ts, down_q, down_s, down_ts,
                  g, u, h, o, n_threads, 0);
}

/* ------------------------------------------------- single NVFP4 quantisation */

/* Largest |v| of a row -> the power-of-two prescale exponent e that puts it in
 * (1344, 2688] (a = m 2^E, 1 <= m < 2: e = 11 - E if m <= 1.3125, else 10 - E),
 * clamped to [-100, 100]; 100 for a row of zeros. */
static int prescale_exp_of(float a)
{
    if (!(a > 0.0f))
        return 100;
    if (!(a < 3.0e38f))
        return -100;
    int ex;
    double f = frexp((double)a, &ex); /* a = f 2^ex, 0.5 <= f < 1 */
    double m = 2.0 * f;
    int E = ex - 1;
    int e = (m <= 1.3125 ? 11 : 10) - E;
    return e < -100 ? -100 : (e > 100 ? 100 : e);
}

/* E4M3 code of the value nearest to a >= 0 (ties: the even code), saturating
 * at 448 (code 0x7E). */
static unsigned e4m3_rne_code(float a)
{
    build_tables();
    if (!(a < 448.0f))
        return 0x7Eu;
    unsigned best = 0;
    double bd = fabs(tab_e4m3[0] - (double)a);
    for (unsigned c = 1; c <= 0x7Eu; ++c) {
        double d = fabs(tab_e4m3[c] - (double)a);
        if (d < bd || (d == bd && (c & 1u) == 0))
            best = c, bd = d;
    }
    return best;
}

/* E2M1 magnitude code of the value nearest to |q| (ties: the even code),
 * saturating at 6; the sign is applied by the caller. */
static unsigned e2m1_rne_mag(float q)
{
    build_tables();
    double m = fabs((double)q);
    if (m >= 6.0)
        return 7u;
    unsigned best = 0;
    double bd = m;
    for (unsigned c = 1; c < 8u; ++c) {
        double d = fabs(tab_e2m1[c] - m);
        if (d < bd || (d == bd && (c & 1u) == 0))
            best = c, bd = d;
    }
    return best;
}

/* One row of n activations (n a multiple of 16) quantised once to NVFP4 and
 * dequantised into out (double): one power-of-two prescale for the row (its
 * largest |v| into (1344, 2688]); per 16-element block the E4M3 scale s = the
 * smallest E4M3 value >= (block max / 6), found as the round-to-nearest-even
 * E4M3 of that quotient, moved up one code when it fell below; each element
 * the round-to-nearest-even E2M1 of (its prescaled value times 1/s).  Every
 * step that decides a code runs in fp32, in this order: v 2^e, max * (1/6),
 * 1/s, (v 2^e) * (1/s).  out = E2M1 value * s * 2^-e. */
static void quant_row_nvfp4(const float *v, int n, double *out)
{
    build_tables();
    float amax = 0.0f;
    for (int i = 0; i < n; ++i)
        amax = fabsf(v[i]) > amax ? fabsf(v[i]) : amax;
    int e = prescale_exp_of(amax);
    volatile float P = ldexpf(1.0f, e);
    const float sixth = 1.0f / 6.0f;
    for (int b = 0; b < n; b += 16) {
        float p[16], bm = 0.0f;
        for (int i = 0; i < 16; ++i) {
            volatile float t = v[b + i] * P;
            p[i] = t;
            bm = fabsf(t) > bm ? fabsf(t) : bm;
        }
        volatile float a = bm * sixth;
        unsigned c = e4m3_rne_code(a);
        if (tab_e4m3[c] < (double)a && c < 0x7Eu)
            ++c;
        double s = tab_e4m3[c];
        if (!(s > 0.0)) {
            for (int i = 0; i < 16; ++i)
                out[b + i] = 0.0;
            continue;
        }
        volatile float inv = 1.0f / (float)s;
        for (int i = 0; i < 16; ++i) {
            volatile float q = p[i] * inv;
            double val = tab_e2m1[e2m1_rne_mag(q)];
            out[b + i] = ldexp((signbit(q) ? -val : val) * s, -e);
        }
    }
}

/* quant_row_nvfp4 as an entry point (n a multiple of 16). */
void oracle_quant_row(const float *v, int n, double *out)
{
    quant_row_nvfp4(v, n, out);
}

/* One (token, expert) pair; act != 0: x already quantised by the caller, h
 * quantised here (expert_pair_q). */
static void expert_pair_mode(int H, int I, int e, const double *xr,
                             const uint8_t *gate_q, const uint8_t *gate_s, const float *gate_ts,
                             const uint8_t *up_q, const uint8_t *up_s, const float *up_ts,
                             const uint8_t *down_q, const uint8_t *down_s, const float *down_ts,
                             double *o, int n_threads, int act)
{
    expert_pair_q(H, I, e, xr, gate_q, gate_s, gate_ts, up_q, up_s, up_ts, down_q, down_s, down_ts,
                  NULL, NULL, NULL, o, n_threads, act);
}

/* ---------------------------------------------------------------- full step */

/* y (double [n_tok, H]) for the tokens listed in `tokens` (NULL: all T, in
 * order), with the three extensions of the step:
 *  - expert range: the routed weight arrays hold experts e_lo .. e_hi-1 only
 *    (array index e - e_lo); a valid id outside the range belongs to another
 *    device's share and contributes nothing here (it is not counted as bad);
 *  - shared expert: when sg_q is not NULL, one always-on expert (arrays
 *    [I, H/2], [I, H/16], [H, I/2], [H, I/16]; s_ts = its gate, up and down
 *    tensor scales) is added to every token's y with weight 1, after the
 *    routed slots;
 *  - act = 1: x and h are quantised once to NVFP4 (quant_row_nvfp4) before
 *    the projections that read them.
 * Returns the number of slots whose id is >= E, or -1 on a bad argument. */
int oracle_moe_forward_ext(int H, int I, int E, int k, int T,
                           const uint16_t *x, const int32_t *ids, const float *w,
                           const uint8_t *gate_q, const uint8_t *gate_s, const float *gate_ts,
                           const uint8_t *up_q, const uint8_t *up_s, const float *up_ts,
                           const uint8_t *down_q, const uint8_t *down_s, const float *down_ts,
                           int e_lo, int e_hi,
                           const uint8_t *sg_q, const uint8_t *sg_s, const uint8_t *su_q, const uint8_t *su_s,
                           const uint8_t *sd_q, const uint8_t *sd_s, const float *s_ts, int act,
                           const int32_t *tokens, int n_tok, double *y, int n_threads)
{
    if (H <= 0 || I <= 0 || E <= 0 || k <= 0 || T < 0 || (H % 16) || (I % 16))
        return -1;
    if (e_lo < 0 || e_hi > E || e_lo >= e_hi)
        return -1;
    if (!tokens)
        n_tok = T;
    double *xr = (double *)malloc(sizeof(double) * (size_t)H);
    double *o = (double *)malloc(sizeof(double) * (size_t)H);
    float *xf = (float *)malloc(sizeof(float) * (size_t)H);
    int bad = 0;
    for (int n = 0; n < n_tok; ++n) {
        int t = tokens ? tokens[n] : n;
        double *yt = y + (size_t)n * H;
        for (int r = 0; r < H; ++r)
            yt[r] = 0.0;
        if (t < 0 || t >= T)
            continue;
        for (int c = 0; c < H; ++c)
            xr[c] = bf16_to_double(x[(size_t)t * H + (size_t)c]);
        if (act) {
            for (int c = 0; c < H; ++c)
                xf[c] = (float)xr[c];
            quant_row_nvfp4(xf, H, xr);
        }
        for (int j = 0; j < k; ++j) {
            int e = ids[(size_t)t * k + (size_t)j];
            if (e < 0)
                continue;
            if (e >= E) {
                ++bad;
                continue;
            }
            if (e < e_lo || e >= e_hi)
                continue;
            expert_pair_mode(H, I, e - e_lo, xr, gate_q, gate_s, gate_ts, up_q, up_s, up_ts,
                             down_q, down_s, down_ts, o, n_threads, act);
            double wj = (double)w[(size_t)t * k + (size_t)j];
            for (int r = 0; r < H; ++r)
                yt[r] += wj * o[r];
        }
        if (sg_q) {
            expert_pair_mode(H, I, 0, xr, sg_q, sg_s, s_ts + 0, su_q, su_s, s_ts + 1, sd_q, sd_s, s_ts + 2,
                             o, n_threads, act);
            for (int r = 0; r < H; ++r)
                yt[r] += o[r];
        }
    }
    free(xr);
    free(o);
    free(xf);
    return bad;
}

/* The plain step: every expert local, no shared expert, exact activations. */
int oracle_moe_forward(int H, int I, int E, int k, int T,
                       const uint16_t *x, const int32_t *ids, const float *w,
                       const uint8_t *gate_q, const uint8_t *gate_s, const float *gate_ts,
                       const uint8_t *up_q, const uint8_t *up_s, const float *up_ts,
                       const uint8_t *down_q, const uint8_t *down_s, const float *down_ts,
                       const int32_t *tokens, int n_tok, double *y, int n_threads)
{
    return oracle_moe_forward_ext(H, I, E, k, T, x, ids, w, gate_q, gate_s, gate_ts, up_q, up_s, up_ts,
                                  down_q, down_s, down_ts, 0, E, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0,
                                  tokens, n_tok, y, n_threads);
}

/* ---------------------------------------------------------------- grouping */

/* Stable counting sort of the P = T*k flat pairs by expert id.
 * counts int32 [E], offsets int32 [E+1], perm int32 [P] (entries past
 * offsets[E] are set to -1).  Returns the number of ids >= E. */
int oracle_group(const int32_t *ids, int P, int E, int32_t *counts, int32_t *offsets, int32_t *perm)
{
    int bad = 0;
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int p = 0; p < P; ++p) {
        int e = ids[p];
        if (e >= E)
            ++bad;
        else if (e >= 0)
            ++counts[e];
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e)
        cursor[e] = offsets[e];
    for (int p = 0; p < P; ++p)
        perm[p] = -1;
    for (int p = 0; p < P; ++p) {
        int e = ids[p];
        if (e >= 0 && e < E)
            perm[cursor[e]++] = p;
    }
    free(cursor);
    return bad;
}

/* ---------------------------------------------------------------- routing */

/* Top-k routing in front of the step: for each token t, the k experts with the
 * largest router logits, in descending order of logit (equal logits: the
 * smaller expert index first; NaN counts as -infinity), and their weights, the
 * softmax over those k logits (in double, then rounded to float).  If the
 * largest selected logit is -infinity the weights are 0; if it is +infinity,
 * the selected +infinity logits share the weight equally and the others get
 * 0 (the softmax's limit as those logits grow together).  This is the router
 * output the input recipe draws at random (k logits, softmax over them); the
 * pages do not describe the router, so it is the plain definition.
 * logits float [T, E]; ids int32 [T, k]; w float [T, k].  Returns -1 on a
 * bad argument (k < 1, k > E, T < 0), else 0. */
int oracle_route(const float *logits, int T, int E, int k, int32_t *ids, float *w)
{
    if (T < 0 || E < 1 || k < 1 || k > E)
        return -1;
    char *taken = (char *)malloc((size_t)E);
    double *sel = (double *)malloc(sizeof(double) * (size_t)k);
    for (int t = 0; t < T; ++t) {
        const float *lt = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            double bv = 0.0;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                double v = isnan(lt[e]) ? -INFINITY : (double)lt[e];
                if (best < 0 || v > bv) {   /* strict: an equal logit keeps the smaller index */
                    best = e;
                    bv = v;
                }
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
            sel[j] = bv;
        }
        /* a +infinity winner: the softmax's limit as the infinite logits grow
         * together, equal weights over the selected +infinity logits */
        double m = sel[0], sum = 0.0;
        for (int j = 0; j < k; ++j)
            sum += (m == -INFINITY) ? 0.0 : (m == INFINITY ? (sel[j] == INFINITY ? 1.0 : 0.0) : exp(sel[j] - m));
        for (int j = 0; j < k; ++j) {
            double ej = (m == INFINITY) ? (sel[j] == INFINITY ? 1.0 : 0.0) : exp(sel[j] - m);
            w[(size_t)t * k + j] = (m == -INFINITY) ? 0.0f : (float)(ej / sum);
        }
    }
    free(taken);
    free(sel);
    return 0;
}
