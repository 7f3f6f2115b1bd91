/*
 * sk_oracle.c -- plain fp64 CPU oracle for length-aware split-KV paged
 * decode/verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [RFC]  vLLM RFC 59111 "NixlConnector: convert standard KV pages to ROCm
 *          AITER shuffled pages on the decode side", Background: standard
 *          pages hold, per head, token rows with K and V side by side
 *          ([H, N, 2*D]), shuffled pages K [H, D/x, N, x] and V
 *          [H, N/x, D, x]; Proposed Change: OCP e4m3fn vs e4m3fnuz, and the
 *          per-block conversion (Convert).
 *   [PR]   SGLang PR 39172 "[AMD] gfx950 assembly attention: length-aware
 *          split-KV for dynamic workload":
 *            Motivation    -- the fixed split max(1, min(64, pow2floor(CUs /
 *                             (bs * kv_heads)))), one work group per
 *                             (segment, sequence, kv head);
 *            Modifications -- the plan: smallest segment length T with total
 *                             segments <= CUs / kv_heads and per-sequence
 *                             segments <= seg_max; work list
 *                             plan[1+i] = seq << 16 | seg, -1 past the end;
 *                             plan[0] = tiles per segment; a per-query-token
 *                             segment count read by the reduce.
 *
 * Everything is evaluated straight from its definition, in double precision,
 * with loops a reader can check by eye.  OpenMP only splits the outer loop over
 * independent output rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SKO_KV_BF16 0
#define SKO_KV_FP8 1

/* bf16 is the upper half of an IEEE-754 binary32. */
double sko_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn": finite, no infinities; the RFC's
 * Proposed Change contrasts it with MI300's e4m3fnuz).  Sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits.  Exponent field 0 is subnormal:
 * (m/8) * 2^-6.  S.1111.111 is NaN; the largest finite value is 448. */
double sko_e4m3fn_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* The e4m3fn code nearest to the binary32 value x, by the same format
 * definition: scan the 127 non-negative finite codes (decoded above) for the
 * closest magnitude, ties going to the even code (even mantissa, as in
 * round-to-nearest-even).  Magnitudes of 448 and above saturate to 448 (0x7E),
 * infinities included; NaN gives 0x7F.  The sign is kept, so -0 and negative
 * values that round to zero give 0x80. */
uint8_t sko_e4m3fn_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const int neg = signbit(x) != 0;
    const double a = fabs((double)x);
    int best = 0x7E;
    if (a < 448.0) {
        double best_d = INFINITY;
        for (int c = 0; c <= 0x7E; ++c) {
            const double d = fabs(sko_e4m3fn_to_double((uint8_t)c) - a);
            if (d < best_d || (d == best_d && (c & 1) == 0)) {
                best_d = d;
                best = c;
            }
        }
    }
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* ---------------------------------------------------------------------------
 * [PR] Motivation: fixed split.  nseg = max(1, min(seg_max, pow2floor(NSM /
 * (bs * kv_heads)))).  pow2floor(x) is the largest power of two <= x and 0
 * when x < 1; taking the integer quotient first does not change it.
 * ------------------------------------------------------------------------ */
int sko_fixed_nseg(int bs, int num_kv_heads, int num_sms, int seg_max)
{
    long long denom = (long long)bs * num_kv_heads;
    long long q = denom > 0 ? (long long)num_sms / denom : 0;
    long long p = 0;
    if (q >= 1) {
        p = 1;
        while (p * 2 <= q)
            p *= 2;
    }
    if (p > seg_max)
        p = seg_max;
    if (p < 1)
        p = 1;
    return (int)p;
}

/* ---------------------------------------------------------------------------
 * [PR] Modifications: the length-aware plan.
 *
 * tiles_s = ceil(L_s / tile).  The budget is B = floor(num_sms / kv_heads)
 * (an integer total <= num_sms/kv_heads is the same as <= B).  T is the
 * smallest t = 1, 2, ... with sum_s ceil(tiles_s / t) <= B and
 * max_s ceil(tiles_s / t) <= seg_max, found by trying every t in order.
 * When no t qualifies (more non-empty sequences than B), T = max_s tiles_s,
 * i.e. one segment per non-empty sequence, the fewest segments possible.
 * With every sequence empty, T = 1 and the work list is empty.
 *
 * Output: plan[0] = T; plan[1 + k] = (s << 16) | g for s ascending, then
 * g ascending, for g < nseg_s = ceil(tiles_s / T); -1 up to plan_capacity;
 * tok_nseg[cu_q[s] + j] = nseg_s for every query token j of sequence s;
 * nseg_out[s] = nseg_s when nseg_out is not NULL.
 * Returns the number of work items, or -1 if plan_capacity is too small.
 * ------------------------------------------------------------------------ */
int sko_plan(const int32_t *seq_lens, const int32_t *cu_q, int bs, int num_kv_heads,
             int num_sms, int seg_max, int tile, int32_t *plan, int plan_capacity,
             int32_t *tok_nseg, int32_t *nseg_out)
{
    int64_t budget = num_kv_heads > 0 ? num_sms / num_kv_heads : 0;
    int64_t max_tiles = 0;
    int64_t t, T = 0;
    int s, k;
    for (s = 0; s < bs; ++s) {
        int64_t tiles = ceil_div64(seq_lens[s], tile);
        if (tiles > max_tiles)
            max_tiles = tiles;
    }
    for (t = 1; t <= (max_tiles > 0 ? max_tiles : 1); ++t) {
        int64_t total = 0, most = 0;
        for (s = 0; s < bs; ++s) {
            int64_t n = ceil_div64(ceil_div64(seq_lens[s], tile), t);
            total += n;
            if (n > most)
                most = n;
        }
        if (total <= budget && most <= seg_max) {
            T = t;
            break;
        }
    }
    if (T == 0)
        T = max_tiles > 0 ? max_tiles : 1;

    k = 0;
    plan[0] = (int32_t)T;
    for (s = 0; s < bs; ++s) {
        int64_t n = ceil_div64(ceil_div64(seq_lens[s], tile), T);
        int64_t g;
        if (nseg_out)
            nseg_out[s] = (int32_t)n;
        for (g = 0; g < n; ++g) {
            if (1 + k >= plan_capacity)
                return -1;
            plan[1 + k] = (int32_t)(((uint32_t)s << 16) | (uint32_t)g);
            ++k;
        }
        if (tok_nseg) {
            int j;
            for (j = cu_q[s]; j < cu_q[s + 1]; ++j)
                tok_nseg[j] = (int32_t)n;
        }
    }
    for (s = 1 + k; s < plan_capacity; ++s)
        plan[s] = -1;
    return k;
}

/* ---------------------------------------------------------------------------
 * Attention definition.
 *
 * Query token t is token j of sequence s (cu_q[s] <= t < cu_q[s+1]) and
 * q_s = cu_q[s+1] - cu_q[s].  Query head hq reads KV head h = hq / G with
 * G = H_q / H_kv.  Key p (0 <= p < L_s) lives in block
 * block_table[s*stride + p/page], row p % page; within that row K is
 * elements [0, D) and V is [D, 2D) ([RFC] Background).  With causal masking
 * token j sees keys p <= L_s - q_s + j (L_s counts this step's tokens).
 *
 *   score_p = sm_scale * k_scale * sum_d q[d] * Kcode_p[d]
 *   out     = v_scale * sum_p softmax(score)_p * Vcode_p
 *   lse     = log sum_p exp(score_p)
 * For bf16 KV the scales are 1.  No visible key: out = 0, lse = -inf.
 * ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q;          /* bf16 bits [NT, H_q, D] */
    const void *kv;             /* [num_blocks, H_kv, page, 2D] bf16 bits or e4m3 codes */
    int kv_dtype;
    double k_scale, v_scale;
    const int32_t *block_table;
    int bt_stride;
    int page;
    const int32_t *seq_lens;
    const int32_t *cu_q;
    int bs, num_q_heads, num_kv_heads, head_dim;
    double sm_scale;
    int causal;
} sko_problem;

static double kv_elem(const sko_problem *P, int s, int h, int p, int d)
{
    int32_t blk = P->block_table[(int64_t)s * P->bt_stride + p / P->page];
    int64_t idx = (((int64_t)blk * P->num_kv_heads + h) * P->page + (p % P->page)) * (2 * P->head_dim) + d;
    if (P->kv_dtype == SKO_KV_FP8)
        return sko_e4m3fn_to_double(((const uint8_t *)P->kv)[idx]);
    return sko_bf16_to_double(((const uint16_t *)P->kv)[idx]);
}

static int seq_of_token(const sko_problem *P, int t)
{
    int s;
    for (s = 0; s < P->bs; ++s)
        if (t >= P->cu_q[s] && t < P->cu_q[s + 1])
            return s;
    return -1;
}

/* Number of keys visible to token j of sequence s: keys [0, n). */
static int visible_keys(const sko_problem *P, int s, int j)
{
    int L = P->seq_lens[s];
    int q = P->cu_q[s + 1] - P->cu_q[s];
    int n = L;
    if (P->causal) {
        n = L - q + j + 1;
        if (n > L)
            n = L;
        if (n < 0)
            n = 0;
    }
    return n;
}

static double score(const sko_problem *P, int t, int hq, int s, int h, int p)
{
    const uint16_t *qrow = P->q + ((int64_t)t * P->num_q_heads + hq) * P->head_dim;
    double acc = 0.0;
    int d;
    for (d = 0; d < P->head_dim; ++d)
        acc += sko_bf16_to_double(qrow[d]) * kv_elem(P, s, h, p, d);
    return P->sm_scale * (P->kv_dtype == SKO_KV_FP8 ? P->k_scale : 1.0) * acc;
}

/* Softmax attention over keys [p0, p1) for one row; writes the un-normalised
 * partial (m, l, o): m = max score, l = sum exp(score - m),
 * o = v_scale * sum exp(score - m) * V.  An empty range gives (-inf, 0, 0). */
static void row_partial(const sko_problem *P, int t, int hq, int p0, int p1,
                        double *m_out, double *l_out, double *o_out)
{
    int s = seq_of_token(P, t);
    int D = P->head_dim;
    int G = P->num_q_heads / P->num_kv_heads;
    int h = hq / G;
    int p, d;
    double m = -INFINITY, l = 0.0;
    double vs = P->kv_dtype == SKO_KV_FP8 ? P->v_scale : 1.0;
    double *sc;
    for (d = 0; d < D; ++d)
        o_out[d] = 0.0;
    if (s < 0 || p1 <= p0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    sc = (double *)malloc(sizeof(double) * (size_t)(p1 - p0));
    for (p = p0; p < p1; ++p) {
        sc[p - p0] = score(P, t, hq, s, h, p);
        if (sc[p - p0] > m)
            m = sc[p - p0];
    }
    for (p = p0; p < p1; ++p) {
        double w = exp(sc[p - p0] - m);
        l += w;
        for (d = 0; d < D; ++d)
            o_out[d] += w * vs * kv_elem(P, s, h, p, D + d);
    }
    free(sc);
    *m_out = m;
    *l_out = l;
}

/* Unsplit attention for the listed rows (row = t * H_q + hq); rows == NULL
 * means every row.  out: [n_rows, D], lse: [n_rows] (either may be NULL). */
void sko_attention(const uint16_t *q, const void *kv, int kv_dtype, double k_scale, double v_scale,
                   const int32_t *block_table, int bt_stride, int page,
                   const int32_t *seq_lens, const int32_t *cu_q, int bs,
                   int num_q_heads, int num_kv_heads, int head_dim, double sm_scale, int causal,
                   const int64_t *rows, int64_t n_rows, double *out, double *lse)
{
    sko_problem P = {q, kv, kv_dtype, k_scale, v_scale, block_table, bt_stride, page,
                     seq_lens, cu_q, bs, num_q_heads, num_kv_heads, head_dim, sm_scale, causal};
    int64_t nt_rows = (int64_t)cu_q[bs] * num_q_heads;
    int64_t count = rows ? n_rows : nt_rows;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < count; ++i) {
        int64_t row = rows ? rows[i] : i;
        int t = (int)(row / num_q_heads), hq = (int)(row % num_q_heads);
        int s = seq_of_token(&P, t);
        int n = s >= 0 ? visible_keys(&P, s, t - cu_q[s]) : 0;
        double m, l;
        double *o = (double *)malloc(sizeof(double) * (size_t)head_dim);
        int d;
        row_partial(&P, t, hq, 0, n, &m, &l, o);
        for (d = 0; d < head_dim; ++d)
            if (out)
                out[i * head_dim + d] = l > 0.0 ? o[d] / l : 0.0;
        if (lse)
            lse[i] = l > 0.0 ? m + log(l) : -INFINITY;
        free(o);
    }
}

/* ---------------------------------------------------------------------------
 * Split evaluation: the same rows computed segment by segment, then merged by
 * log-sum-exp.  Segment g of sequence s covers keys
 * [g*T, min((g+1)*T, L_s)) with T = seg_tiles[s] * tile tokens, for
 * g < nseg[s].  The partial of each (token, segment, head) is written to
 * part_o [NT, seg_max, H_q, D], part_m / part_l [NT, seg_max, H_q] (any may
 * be NULL), then merged:
 *   M = max_g m_g,  Lambda = sum_g l_g exp(m_g - M),
 *   out = sum_g o_g exp(m_g - M) / Lambda,   lse = M + log Lambda.
 * Lambda = 0 gives out = 0 and lse = -inf.
 * ------------------------------------------------------------------------ */
void sko_attention_split(const uint16_t *q, const void *kv, int kv_dtype, double k_scale, double v_scale,
                         const int32_t *block_table, int bt_stride, int page,
                         const int32_t *seq_lens, const int32_t *cu_q, int bs,
                         int num_q_heads, int num_kv_heads, int head_dim, double sm_scale, int causal,
                         const int32_t *nseg, const int32_t *seg_tiles, int tile, int seg_max,
                         double *part_o, double *part_m, double *part_l, double *out, double *lse)
{
    sko_problem P = {q, kv, kv_dtype, k_scale, v_scale, block_table, bt_stride, page,
                     seq_lens, cu_q, bs, num_q_heads, num_kv_heads, head_dim, sm_scale, causal};
    int64_t nrows = (int64_t)cu_q[bs] * num_q_heads;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = 0; i < nrows; ++i) {
        int t = (int)(i / num_q_heads), hq = (int)(i % num_q_heads);
        int s = seq_of_token(&P, t);
        int D = head_dim;
        int n_vis = s >= 0 ? visible_keys(&P, s, t - cu_q[s]) : 0;
        int ns = s >= 0 ? nseg[s] : 0;
        int64_t T = s >= 0 ? (int64_t)seg_tiles[s] * tile : 0;
        double *mg = (double *)malloc(sizeof(double) * (size_t)(ns > 0 ? ns : 1));
        double *lg = (double *)malloc(sizeof(double) * (size_t)(ns > 0 ? ns : 1));
        double *og = (double *)malloc(sizeof(double) * (size_t)(ns > 0 ? ns : 1) * D);
        double M = -INFINITY, Lam = 0.0;
        int g, d;
        for (g = 0; g < ns; ++g) {
            int64_t a = g * T, b = (g + 1) * T;
            if (b > seq_lens[s])
                b = seq_lens[s];
            if (b > n_vis)
                b = n_vis;
            row_partial(&P, t, hq, (int)a, (int)(b > a ? b : a), &mg[g], &lg[g], &og[(int64_t)g * D]);
            if (part_m)
                part_m[((int64_t)t * seg_max + g) * num_q_heads + hq] = mg[g];
            if (part_l)
                part_l[((int64_t)t * seg_max + g) * num_q_heads + hq] = lg[g];
            if (part_o)
                for (d = 0; d < D; ++d)
                    part_o[(((int64_t)t * seg_max + g) * num_q_heads + hq) * D + d] = og[(int64_t)g * D + d];
            if (mg[g] > M)
                M = mg[g];
        }
        for (g = 0; g < ns; ++g)
            if (lg[g] > 0.0)
                Lam += lg[g] * exp(mg[g] - M);
        for (d = 0; d < D; ++d) {
            double acc = 0.0;
            for (g = 0; g < ns; ++g)
                if (lg[g] > 0.0)
                    acc += og[(int64_t)g * D + d] * exp(mg[g] - M);
            if (out)
                out[i * D + d] = Lam > 0.0 ? acc / Lam : 0.0;
        }
        if (lse)
            lse[i] = Lam > 0.0 ? M + log(Lam) : -INFINITY;
        free(mg);
        free(lg);
        free(og);
    }
}

/* ---------------------------------------------------------------------------
 * [PR] Modifications (the reduce reads only its token's segment count): merge
 * given partials.  n = tok_nseg[t] when tok_nseg is not NULL, else fixed_nseg.
 * Partials are float32 in the layout above; a segment with l = 0 contributes
 * nothing.
 * ------------------------------------------------------------------------ */
void sko_merge(const float *part_o, const float *part_m, const float *part_l,
               const int32_t *tok_nseg, int fixed_nseg, int num_tokens, int num_q_heads,
               int head_dim, int seg_max, double *out, double *lse)
{
    int64_t nrows = (int64_t)num_tokens * num_q_heads;
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int t = (int)(i / num_q_heads), hq = (int)(i % num_q_heads);
        int n = tok_nseg ? tok_nseg[t] : fixed_nseg;
        double M = -INFINITY, Lam = 0.0;
        int g, d;
        for (g = 0; g < n; ++g) {
            int64_t k = ((int64_t)t * seg_max + g) * num_q_heads + hq;
            if (part_l[k] > 0.0f && (double)part_m[k] > M)
                M = part_m[k];
        }
        for (g = 0; g < n; ++g) {
            int64_t k = ((int64_t)t * seg_max + g) * num_q_heads + hq;
            if (part_l[k] > 0.0f)
                Lam += (double)part_l[k] * exp((double)part_m[k] - M);
        }
        for (d = 0; d < head_dim; ++d) {
            double acc = 0.0;
            for (g = 0; g < n; ++g) {
                int64_t k = ((int64_t)t * seg_max + g) * num_q_heads + hq;
                if (part_l[k] > 0.0f)
                    acc += (double)part_o[k * head_dim + d] * exp((double)part_m[k] - M);
            }
            out[i * head_dim + d] = Lam > 0.0 ? acc / Lam : 0.0;
        }
        if (lse)
            lse[i] = Lam > 0.0 ? M + log(Lam) : -INFINITY;
    }
}

/* ---------------------------------------------------------------------------
 * [RFC] Background: the KV write of the backends that keep standard pages.
 * Token t's K and V rows for KV head h land side by side in row
 * (slot % page) of block (slot / page), slot = slot_mapping[t]:
 *   pages[blk][h][off][0:D] = K[t][h][:],  pages[blk][h][off][D:2D] = V[t][h][:].
 * A negative slot marks a token without a cache slot: nothing is written for
 * it, nor for a slot past the last block.  Tokens are taken in order, so a
 * slot given twice ends with the later token (the GPU path leaves that case
 * undefined).  bf16 pages receive the input bits unchanged; e4m3 pages
 * receive sko_e4m3fn_encode(x / scale), the quotient rounded to binary32
 * (IEEE division, the precision the CUDA path divides in), with k_scale for
 * K and v_scale for V. */
void sko_reshape_and_cache(const uint16_t *key, const uint16_t *value, const int64_t *slot_mapping,
                           int num_tokens, int num_kv_heads, int head_dim, void *kv_pages,
                           int kv_dtype, float k_scale, float v_scale, int64_t num_blocks, int page)
{
    const int64_t row_elems = 2 * (int64_t)head_dim;
    for (int t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        const int64_t blk = slot / page, off = slot % page;
        if (blk >= num_blocks)
            continue;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t row = ((blk * num_kv_heads + h) * page + off) * row_elems;
            const int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                if (kv_dtype == SKO_KV_BF16) {
                    uint16_t *pg = (uint16_t *)kv_pages;
                    pg[row + d] = key[src + d];
                    pg[row + head_dim + d] = value[src + d];
                } else {
                    uint8_t *pg = (uint8_t *)kv_pages;
                    const float kq = (float)sko_bf16_to_double(key[src + d]) / k_scale;
                    const float vq = (float)sko_bf16_to_double(value[src + d]) / v_scale;
                    pg[row + d] = sko_e4m3fn_encode(kq);
                    pg[row + head_dim + d] = sko_e4m3fn_encode(vq);
                }
            }
        }
    }
}

/* ---------------------------------------------------------------------------
 * [RFC] Proposed Change, step 4 (Convert): the decode side's per-block view and
 * permute from standard pages to AITER's shuffled pages, with x = 16 / element
 * size (8 for bf16, 16 for e4m3).  For block blk, head h, token row n and
 * dimension d of K = page[..., 0:D) and V = page[..., D:2D):
 *   k_shuf[blk][h][d / x][n][d % x] = K[blk][h][n][d]     (k_shuf [NB, H, D/x, N, x])
 *   v_shuf[blk][h][n / x][d][n % x] = V[blk][h][n][d]     (v_shuf [NB, H, N/x, D, x])
 * for every block in block_ids (all blocks when block_ids is NULL); other
 * blocks of the outputs are left alone, as are ids outside [0, num_blocks).
 * Pure data movement: elements are copied as elem_size-byte units. */
void sko_std_to_shuffled(const void *kv_pages, int elem_size, const int32_t *block_ids, int num_ids,
                         int64_t num_blocks, int num_kv_heads, int head_dim, int page, void *k_shuf,
                         void *v_shuf)
{
    const int x = 16 / elem_size;
    const int n_ids = block_ids ? num_ids : (int)num_blocks;
    const uint8_t *src = (const uint8_t *)kv_pages;
    uint8_t *ko = (uint8_t *)k_shuf, *vo = (uint8_t *)v_shuf;
    for (int i = 0; i < n_ids; ++i) {
        const int64_t blk = block_ids ? block_ids[i] : i;
        if (blk < 0 || blk >= num_blocks)
            continue;
        for (int h = 0; h < num_kv_heads; ++h) {
            const int64_t bh = blk * num_kv_heads + h;
            for (int n = 0; n < page; ++n) {
                for (int d = 0; d < head_dim; ++d) {
                    const int64_t k_src = ((bh * page + n) * 2 * head_dim + d) * elem_size;
                    const int64_t v_src = ((bh * page + n) * 2 * head_dim + head_dim + d) * elem_size;
                    const int64_t k_dst = (((bh * (head_dim / x) + d / x) * page + n) * x + d % x) * elem_size;
                    const int64_t v_dst = (((bh * (page / x) + n / x) * head_dim + d) * x + n % x) * elem_size;
                    memcpy(ko + k_dst, src + k_src, (size_t)elem_size);
                    memcpy(vo + v_dst, src + v_src, (size_t)elem_size);
                }
            }
        }
    }
}

/* Threads the OpenMP loops above use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
#endif
int sko_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the thread count of the loops above (n <= 0: every processor); a no-op
 * without OpenMP.  Timing only: the results do not depend on it. */
void sko_set_num_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}
