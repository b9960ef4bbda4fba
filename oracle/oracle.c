/*
 * oracle.c -- plain, slow, single-threaded CPU reference of the global-retrieval
 * half of the hybrid attention described for GLM-5.3-Flash.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this code.  The CUDA library shares nothing with it
 * (no header, helper, table or constant) and never calls it.
 *
 * What it computes, step by step, in the order of the DSA layer diagram
 * (page "G2C Brief -- GLM-5.3-Flash", section "DSA keeps selected global access
 * in eleven layers"): full token history -> IndexPool -> learned sparse
 * selection (top-k) -> attention over the selected history.
 *
 *   pool    kbar[b,g,:] = sum_{j<P} alpha[b,g,j] * k[b, P*g+j, :]
 *           ("four indexer key vectors into one via weighted pooling";
 *            reading notes "GLM-5.3-Flash: Hybrid Attention, IndexPool, and
 *            Vision-in-the-Loop", section 2 sub-head "IndexPool").
 *   score   s[b,t,g] = sum_h w[b,t,h] * max(0, q[b,t,h,:] . kbar[b,g,:])
 *           (the lightweight multi-head indexer; the pages name it only by
 *            its DSA-indexer lineage, section 2 of the reading notes, and give
 *            no formula, so this is the DSA indexer's ReLU-weighted form).
 *   mask    decode: every complete group g < L_b/P is visible; chunked
 *           prefill: group g is visible to the query at absolute position p
 *           iff P*g + P - 1 <= p (only complete past groups).
 *   select  the k visible groups of largest s; equal scores -> lower g first;
 *           emitted in ascending g, padded with -1 when fewer than k are
 *           visible ("learned sparse selection (top 2048)", index_topk 2048 =
 *           512 groups of 4 tokens).
 *   attend  softmax attention of every query head over the P*k tokens the
 *           selected groups cover, one shared K/V head ("attention over
 *           selected history").
 *
 * Arithmetic: every product and sum in double; each result rounded once to
 * its storage type (bf16 round-to-nearest-even from the exact binary value,
 * fp32 by C's double->float conversion).  Compile with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 --- */

static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Nearest bf16 to x (8 significant bits, ties to even), from the format's
 * definition: scale |x| so that its quantum becomes 1, round to an integer
 * with ties to even (rint in the default rounding mode), scale back. */
uint16_t oracle_bf16_from_double(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80u;
    int e;
    frexp(a, &e);             /* a = f * 2^e, f in [0.5, 1)          */
    int qe = e - 8;           /* quantum of an 8-significant-bit value */
    if (qe < -133)
        qe = -133;            /* bf16 subnormal quantum 2^-133          */
    double r = rint(ldexp(a, -qe));
    double y = ldexp(r, qe);
    if (y >= 0x1p128)
        return sign | 0x7F80u;
    float f = (float)y;       /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFFu);
}

/* ---------------------------------------------------------------- pool --- */

/* The pooled sum is formed exactly, then rounded once.  A product of an fp32
 * weight (at most 24 significant bits) and a bf16 key (at most 8) is an
 * integer m with |m| < 2^32 times 2^e, -282 <= e <= 224; a sum of P <= 8 such
 * products is held exactly in a two's-complement integer of WIDE_LIMBS 64-bit
 * limbs whose lowest bit weighs 2^WIDE_E0 (bits up to 2^(WIDE_E0 + 640)). */
#define WIDE_LIMBS 10
#define WIDE_E0 (-288)

typedef struct {
    uint64_t w[WIDE_LIMBS];
} wide_int;

static void wide_negate(wide_int *a)
{
    int carry = 1;
    for (int i = 0; i < WIDE_LIMBS; ++i) {
        a->w[i] = ~a->w[i] + (uint64_t)carry;
        carry = carry && a->w[i] == 0;
    }
}

/* a += m * 2^e  (|m| < 2^63, e >= WIDE_E0, m * 2^e inside the range above) */
static void wide_add(wide_int *a, int64_t m, int e)
{
    if (m == 0)
        return;
    wide_int t;
    memset(&t, 0, sizeof t);
    uint64_t mag = m < 0 ? (uint64_t)(-m) : (uint64_t)m;
    int pos = e - WIDE_E0, limb = pos / 64, sh = pos % 64;
    t.w[limb] = mag << sh;
    if (sh && limb + 1 < WIDE_LIMBS)
        t.w[limb + 1] = mag >> (64 - sh);
    if (m < 0)
        wide_negate(&t);
    uint64_t carry = 0;
    for (int i = 0; i < WIDE_LIMBS; ++i) {
        uint64_t s = a->w[i] + t.w[i];
        uint64_t c1 = s < t.w[i];
        uint64_t s2 = s + carry;
        uint64_t c2 = s2 < s;
        a->w[i] = s2;
        carry = c1 | c2;
    }
}

static int wide_bit(const wide_int *a, int i)
{
    return (int)((a->w[i / 64] >> (i % 64)) & 1u);
}

/* a finite nonzero float as m * 2^e with m an odd integer of at most 24 bits
 * (so e is the weight of its lowest set bit: e >= -149 for fp32, >= -133 for
 * bf16); zero as m = 0 */
static void split_float(float f, int64_t *m, int *e)
{
    *m = 0;
    *e = 0;
    if (f == 0.0f)
        return;
    int ex;
    double fr = frexp((double)f, &ex);  /* f = fr * 2^ex, 0.5 <= |fr| < 1 */
    int64_t mm = (int64_t)ldexp(fr, 24);  /* exact */
    int ee = ex - 24;
    while ((mm & 1) == 0) {
        mm /= 2;
        ee += 1;
    }
    *m = mm;
    *e = ee;
}

/* Nearest bf16 of the exact integer value (ties to even): take the 8 bits
 * from the leading one (fewer below the subnormal quantum 2^-133), then the
 * first bit below them and whether any lower bit is set. */
static uint16_t wide_to_bf16(const wide_int *acc)
{
    wide_int a = *acc;
    uint16_t sign = 0;
    if (a.w[WIDE_LIMBS - 1] >> 63) {
        sign = 0x8000u;
        wide_negate(&a);
    }
    int top = -1;
    for (int i = WIDE_LIMBS * 64 - 1; i >= 0; --i)
        if (wide_bit(&a, i)) {
            top = i;
            break;
        }
    if (top < 0)
        return 0;                       /* an exact zero sum is +0 */
    int qe = top + WIDE_E0 - 7;         /* quantum of 8 significant bits */
    if (qe < -133)
        qe = -133;
    int cut = qe - WIDE_E0;             /* bit index of the quantum (> 0) */
    uint64_t r = 0;
    for (int i = top; i >= cut; --i)
        r = 2 * r + (uint64_t)wide_bit(&a, i);
    int half = wide_bit(&a, cut - 1), sticky = 0;
    for (int i = cut - 2; i >= 0 && !sticky; --i)
        sticky = wide_bit(&a, i);
    if (half && (sticky || (r & 1u)))
        r += 1;
    double y = ldexp((double)r, qe);
    if (y >= 0x1p128)
        return sign | 0x7F80u;
    float f = (float)y;                 /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFFu);
}

/* IndexPool over every complete group of every sequence.
 * k_idx [B][*][d] (batch stride sk_b elements), pool_w [B][*][P] (stride sw_b),
 * k_pooled [B][*][d] (stride sp_b).  Groups g >= seq_len[b]/P are untouched.
 * Finite inputs: the sum is exact and rounded once; a non-finite weight or
 * key takes IEEE double arithmetic (inf or NaN out). */
void oracle_pool_keys(const uint16_t *k_idx, int64_t sk_b, const float *pool_w, int64_t sw_b,
                      const int32_t *seq_len, int B, int d, int P,
                      uint16_t *k_pooled, int64_t sp_b)
{
    for (int b = 0; b < B; ++b) {
        int64_t G = seq_len[b] / P;
        for (int64_t g = 0; g < G; ++g) {
            const float *alpha = pool_w + b * sw_b + g * P;
            for (int i = 0; i < d; ++i) {
                wide_int acc;
                memset(&acc, 0, sizeof acc);
                double s = 0.0;
                int finite = 1;
                for (int j = 0; j < P; ++j) {
                    double kv = bf16_value(k_idx[b * sk_b + (P * g + j) * (int64_t)d + i]);
                    double aj = (double)alpha[j];
                    s += aj * kv;
                    if (!isfinite(aj) || !isfinite(kv)) {
                        finite = 0;
                        continue;
                    }
                    int64_t ma, mk;
                    int ea, ek;
                    split_float((float)aj, &ma, &ea);
                    split_float((float)kv, &mk, &ek);
                    wide_add(&acc, ma * mk, ea + ek);
                }
                k_pooled[b * sp_b + g * (int64_t)d + i] =
                    finite ? wide_to_bf16(&acc) : oracle_bf16_from_double(s);
            }
        }
    }
}

/* ------------------------------------------------------------- visible --- */

/* Number of visible groups for query t of sequence b (a prefix [0, n)). */
static int64_t visible_groups(const int32_t *seq_len, const int32_t *q_pos, int b, int T, int t, int P)
{
    int64_t n = seq_len[b] / P;
    if (q_pos) {
        int64_t p = q_pos[(int64_t)b * T + t];
        int64_t m = (p + 1) / P;   /* groups whose last token P*g+P-1 <= p */
        if (p < 0)
            m = 0;
        if (m < n)
            n = m;
    }
    return n;
}

void oracle_visible_counts(const int32_t *seq_len, const int32_t *q_pos, int B, int T, int P,
                           int32_t *n_valid)
{
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            n_valid[(int64_t)b * T + t] = (int32_t)visible_groups(seq_len, q_pos, b, T, t, P);
}

/* --------------------------------------------------------------- score --- */

/* s[b][t][g] for g < visible count; -inf elsewhere.  -0 is stored as +0. */
void oracle_index_scores(const uint16_t *q_idx, const float *w_head,
                         const uint16_t *k_pooled, int64_t sp_b,
                         const int32_t *seq_len, const int32_t *q_pos,
                         int B, int T, int H_i, int d, int P, int64_t G_max, float *scores)
{
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t n = visible_groups(seq_len, q_pos, b, T, t, P);
            const uint16_t *qt = q_idx + ((int64_t)b * T + t) * H_i * d;
            const float *wt = w_head + ((int64_t)b * T + t) * H_i;
            float *st = scores + ((int64_t)b * T + t) * G_max;
            for (int64_t g = 0; g < G_max; ++g) {
                if (g >= n) {
                    st[g] = -INFINITY;
                    continue;
                }
                const uint16_t *kg = k_pooled + b * sp_b + g * d;
                double s = 0.0;
                for (int h = 0; h < H_i; ++h) {
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i)
                        dot += bf16_value(qt[h * d + i]) * bf16_value(kg[i]);
                    double relu = dot > 0.0 ? dot : 0.0;
                    s += (double)wt[h] * relu;
                }
                float f = (float)s;
                st[g] = (f == 0.0f) ? 0.0f : f;
            }
        }
    }
}

/* -------------------------------------------------------------- select --- */

typedef struct {
    float s;
    int32_t g;
} cand_t;

/* larger score first; equal scores (including -0 == +0): lower index first */
static int by_score_desc(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->s > b->s)
        return -1;
    if (a->s < b->s)
        return 1;
    return (a->g < b->g) ? -1 : (a->g > b->g);
}

static int by_index_asc(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Per row: the min(k, n_valid) visible groups of largest score, ascending by
 * index, then -1 padding.  Rows are [rows][G_max]; valid groups are the prefix
 * [0, n_valid[row]). */
void oracle_topk(const float *scores, const int32_t *n_valid, int64_t rows, int64_t G_max, int k,
                 int32_t *idx)
{
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(G_max > 0 ? G_max : 1));
    for (int64_t r = 0; r < rows; ++r) {
        int64_t n = n_valid[r];
        if (n > G_max)
            n = G_max;
        const float *sr = scores + r * G_max;
        for (int64_t g = 0; g < n; ++g) {
            c[g].s = sr[g];
            c[g].g = (int32_t)g;
        }
        qsort(c, (size_t)n, sizeof(cand_t), by_score_desc);
        int64_t m = n < k ? n : k;
        int32_t *out = idx + r * k;
        for (int64_t j = 0; j < m; ++j)
            out[j] = c[j].g;
        qsort(out, (size_t)m, sizeof(int32_t), by_index_asc);
        for (int64_t j = m; j < k; ++j)
            out[j] = -1;
    }
    free(c);
}

/* -------------------------------------------------------------- attend --- */

/* For each (b, t) and query head h: softmax over the tokens of the selected
 * groups (entries < 0 or >= seq_len[b]/P are skipped), one shared K/V head.
 * out [B][T][H_q][d_v] bf16, lse [B][T][H_q] natural-log sum of exp (nullable).
 * No selected token: output 0, lse -inf. */
void oracle_sparse_attn(const uint16_t *q, const uint16_t *K, int64_t sK_b,
                        const uint16_t *V, int64_t sV_b, const int32_t *seq_len,
                        const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v, int P, int k,
                        double scale, uint16_t *out, float *lse)
{
    int64_t max_tok = (int64_t)k * P;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_tok > 0 ? max_tok : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(max_tok > 0 ? max_tok : 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)d_v);
    for (int b = 0; b < B; ++b) {
        int64_t G = seq_len[b] / P;
        for (int t = 0; t < T; ++t) {
            const int32_t *sel = idx + ((int64_t)b * T + t) * k;
            int64_t n = 0;
            for (int j = 0; j < k; ++j) {
                int64_t g = sel[j];
                if (g < 0 || g >= G)
                    continue;
                for (int i = 0; i < P; ++i)
                    tok[n++] = P * g + i;
            }
            for (int h = 0; h < H_q; ++h) {
                const uint16_t *qh = q + (((int64_t)b * T + t) * H_q + h) * d_qk;
                uint16_t *oh = out + (((int64_t)b * T + t) * H_q + h) * d_v;
                float *lh = lse ? lse + ((int64_t)b * T + t) * H_q + h : NULL;
                if (n == 0) {
                    for (int i = 0; i < d_v; ++i)
                        oh[i] = 0;
                    if (lh)
                        *lh = -INFINITY;
                    continue;
                }
                double m = -INFINITY;
                for (int64_t j = 0; j < n; ++j) {
                    const uint16_t *kj = K + b * sK_b + tok[j] * d_qk;
                    double dot = 0.0;
                    for (int i = 0; i < d_qk; ++i)
                        dot += bf16_value(qh[i]) * bf16_value(kj[i]);
                    z[j] = scale * dot;
                    if (z[j] > m)
                        m = z[j];
                }
                double l = 0.0;
                for (int i = 0; i < d_v; ++i)
                    o[i] = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    double p = exp(z[j] - m);
                    l += p;
                    const uint16_t *vj = V + b * sV_b + tok[j] * d_v;
                    for (int i = 0; i < d_v; ++i)
                        o[i] += p * bf16_value(vj[i]);
                }
                for (int i = 0; i < d_v; ++i)
                    oh[i] = oracle_bf16_from_double(o[i] / l);
                if (lh)
                    *lh = (float)(m + log(l));
            }
        }
    }
    free(o);
    free(z);
    free(tok);
}

/* ---------------------------------------------------------- whole step --- */

/* One retrieval step over already pooled keys: score -> select -> attend.
 * scores [B][T][G_max] and idx [B][T][k] are outputs (scores is also the
 * working buffer of the selection). */
void oracle_retrieval_step(const uint16_t *q_idx, const float *w_head,
                           const uint16_t *k_pooled, int64_t sp_b,
                           const uint16_t *q, const uint16_t *K, int64_t sK_b,
                           const uint16_t *V, int64_t sV_b,
                           const int32_t *seq_len, const int32_t *q_pos,
                           int B, int T, int H_i, int d_idx, int P, int64_t G_max, int k,
                           int H_q, int d_qk, int d_v, double scale,
                           float *scores, int32_t *idx, uint16_t *out, float *lse)
{
    int32_t *n_valid = (int32_t *)malloc(sizeof(int32_t) * (size_t)B * (size_t)T);
    oracle_index_scores(q_idx, w_head, k_pooled, sp_b, seq_len, q_pos, B, T, H_i, d_idx, P,
                        G_max, scores);
    oracle_visible_counts(seq_len, q_pos, B, T, P, n_valid);
    oracle_topk(scores, n_valid, (int64_t)B * T, G_max, k, idx);
    oracle_sparse_attn(q, K, sK_b, V, sV_b, seq_len, idx, B, T, H_q, d_qk, d_v, P, k, scale,
                       out, lse);
    free(n_valid);
}

/* ---------------------------------------------------------------- FP8 --- */
/*
 * FP8 pooled indexer keys and queries (a next step of the path, not yet on
 * the GPU).  The pages say only that the serving stack quantizes its caches
 * per tier to INT8, FP8 or BF16 (reading notes, section "The serving stack";
 * G2C Brief, section "Serving: the architecture is only half the efficiency
 * claim").  Format and scaling here are readings:
 *   e4m3   the OCP 8-bit float E4M3: sign, 4 exponent bits (bias 7), 3
 *          mantissa bits, no infinities, S.1111.111 is NaN; largest finite
 *          magnitude 448 = 1.75 * 2^8, smallest normal 2^-6, subnormals
 *          m * 2^-9 (m = 1..7).
 *   round  to the nearest representable value, ties to the even code,
 *          saturating at +-448.
 *   scale  one per 64-element row: amax / 448 rounded to fp32 (0 for an
 *          all-zero row); code_i = e4m3(x_i / scale).
 *   score  s = sum_h w_h * max(0, sq_h * sk_g * sum_i v(cq_hi) * v(ck_gi)),
 *          every step in double, rounded once to fp32, with the visibility
 *          rule of the bf16 score.
 */
double oracle_e4m3_value(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* exhaustive nearest over the 127 codes 0x00..0x7E (0 .. 448) */
uint8_t oracle_e4m3_from_double(double x)
{
    const uint8_t sign = (x < 0.0 || (x == 0.0 && signbit(x))) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    uint8_t best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double d = fabs(oracle_e4m3_value((uint8_t)c) - a);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            bd = d;
            best = (uint8_t)c;
        }
    }
    return sign | best;
}

void oracle_quantize_rows_e4m3(const uint16_t *x, int64_t rows, int d, uint8_t *code, float *scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * d;
        double amax = 0.0;
        for (int i = 0; i < d; ++i) {
            const double a = fabs(bf16_value(xr[i]));
            if (a > amax) amax = a;
        }
        const float sc = (float)(amax / 448.0);
        scale[r] = sc;
        for (int i = 0; i < d; ++i)
            code[r * d + i] = sc == 0.0f ? 0 : oracle_e4m3_from_double(bf16_value(xr[i]) / (double)sc);
    }
}

void oracle_index_scores_e4m3(const uint8_t *cq, const float *sq, const float *w_head,
                              const uint8_t *ck, const float *sk, int64_t sp_b,
                              const int32_t *seq_len, const int32_t *q_pos,
                              int B, int T, int H_i, int d, int P, int64_t G_max, float *scores)
{
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            const int64_t n = visible_groups(seq_len, q_pos, b, T, t, P);
            const int64_t bt = (int64_t)b * T + t;
            float *st = scores + bt * G_max;
            for (int64_t g = 0; g < G_max; ++g) {
                if (g >= n) {
                    st[g] = -INFINITY;
                    continue;
                }
                const int64_t kr = (b * sp_b) / d + g;  /* the key's row */
                double s = 0.0;
                for (int h = 0; h < H_i; ++h) {
                    const int64_t qr = bt * H_i + h;
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i)
                        dot += oracle_e4m3_value(cq[qr * d + i]) * oracle_e4m3_value(ck[kr * d + i]);
                    dot *= (double)sq[qr] * (double)sk[kr];
                    s += (double)w_head[qr] * (dot > 0.0 ? dot : 0.0);
                }
                const float f = (float)s;
                st[g] = (f == 0.0f) ? 0.0f : f;
            }
        }
    }
}

/* -------------------------------------------------- FP8 (E4M3) K/V cache --- */

/* Attention as oracle_sparse_attn, over a K/V cache held as E4M3 codes with one
 * fp32 scale per token row (the same format as the FP8 pooled keys: scale =
 * amax / 448, see oracle_quantize_rows_e4m3).  The serving stack of the
 * reading notes quantizes caches per tier to INT8, FP8 or BF16 ("The serving
 * stack"); the element value is e4m3(code) * scale, exact in double:
 *
 *   z_j = scale_softmax * sum_i q_i * e4m3(kc[j][i]) * ks[j]
 *   out = sum_j softmax_j(z) * e4m3(vc[j][:]) * vs[j]
 *
 * kc [B][*][d_qk] and vc [B][*][d_v] codes with batch strides skc_b, svc_b
 * elements; ks, vs [B][*] with batch strides sks_b, svs_b. */
void oracle_sparse_attn_e4m3kv(const uint16_t *q, const uint8_t *kc, int64_t skc_b,
                               const float *ks, int64_t sks_b, const uint8_t *vc, int64_t svc_b,
                               const float *vs, int64_t svs_b, const int32_t *seq_len,
                               const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                               int P, int k, double scale, uint16_t *out, float *lse)
{
    int64_t max_tok = (int64_t)k * P;
    int64_t *tok = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_tok > 0 ? max_tok : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(max_tok > 0 ? max_tok : 1));
    double *o = (double *)malloc(sizeof(double) * (size_t)d_v);
    for (int b = 0; b < B; ++b) {
        const int64_t G = seq_len[b] / P;
        for (int t = 0; t < T; ++t) {
            const int32_t *sel = idx + ((int64_t)b * T + t) * k;
            int64_t n = 0;
            for (int j = 0; j < k; ++j) {
                const int64_t g = sel[j];
                if (g < 0 || g >= G)
                    continue;
                for (int i = 0; i < P; ++i)
                    tok[n++] = P * g + i;
            }
            for (int h = 0; h < H_q; ++h) {
                const uint16_t *qh = q + (((int64_t)b * T + t) * H_q + h) * d_qk;
                uint16_t *oh = out + (((int64_t)b * T + t) * H_q + h) * d_v;
                float *lh = lse ? lse + ((int64_t)b * T + t) * H_q + h : NULL;
                if (n == 0) {
                    for (int i = 0; i < d_v; ++i)
                        oh[i] = 0;
                    if (lh)
                        *lh = -INFINITY;
                    continue;
                }
                double m = -INFINITY;
                for (int64_t j = 0; j < n; ++j) {
                    const uint8_t *kj = kc + b * skc_b + tok[j] * d_qk;
                    const double sk = (double)ks[b * sks_b + tok[j]];
                    double dot = 0.0;
                    for (int i = 0; i < d_qk; ++i)
                        dot += bf16_value(qh[i]) * (oracle_e4m3_value(kj[i]) * sk);
                    z[j] = dot * scale;
                    if (z[j] > m)
                        m = z[j];
                }
                double l = 0.0;
                for (int i = 0; i < d_v; ++i)
                    o[i] = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    const double p = exp(z[j] - m);
                    l += p;
                    const uint8_t *vj = vc + b * svc_b + tok[j] * d_v;
                    const double sv = (double)vs[b * svs_b + tok[j]];
                    for (int i = 0; i < d_v; ++i)
                        o[i] += p * (oracle_e4m3_value(vj[i]) * sv);
                }
                const double lsum = l;
                for (int i = 0; i < d_v; ++i)
                    oh[i] = oracle_bf16_from_double(o[i] / lsum);
                if (lh)
                    *lh = (float)(log(l) + m);
            }
        }
    }
    free(o);
    free(z);
    free(tok);
}

/* ------------------------------------------------------- INT8 K/V cache --- */

/* The INT8 tier of the same serving stack (reading notes, "The serving
 * stack": caches quantized per tier to INT8, FP8 or BF16; no format given).
 * Readings:
 *   code   a signed 8-bit integer in [-127, 127] (symmetric, -128 unused)
 *   scale  one per token row: amax / 127 rounded to fp32 (0 for an all-zero
 *          row, whose codes are all 0)
 *   round  code_i = the integer nearest to x_i / scale, ties to the even
 *          integer; |x_i| <= amax keeps it within +-127
 *   value  code * scale, exact in double (8 by 24 significant bits)
 * The nearest integer is found by trying every magnitude 0..127 against |x|
 * (c * scale is exact in double, and so is its distance to |x| wherever two
 * candidates come close). */
double oracle_i8_value(int8_t c, float scale)
{
    return (double)c * (double)scale;
}

int8_t oracle_i8_from_double(double x, float scale)
{
    const double a = fabs(x);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 127; ++c) {
        const double d = fabs((double)c * (double)scale - a);
        if (d < bd || (d == bd && c % 2 == 0)) {
            bd = d;
            best = c;
        }
    }
    return (int8_t)(x < 0.0 ? -best : best);
}

void oracle_quantize_rows_i8(const uint16_t *x, int64_t rows, int d, int8_t *code, float *scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * d;
        double amax = 0.0;
        for (int i = 0; i < d; ++i) {
            const double a = fabs(bf16_value(xr[i]));
            if (a > amax) amax = a;
        }
        const float sc = (float)(amax / 127.0);
        scale[r] = sc;
        for (int i = 0; i < d; ++i)
            code[r * d + i] = sc == 0.0f ? 0 : oracle_i8_from_double(bf16_value(xr[i]), sc);
    }
}

/* Attention over an INT8 K/V cache, the definition written out:
 *
 *   z_j = scale_softmax * sum_i q_i * (kc[j][i] * ks[j])
 *   out = sum_j softmax_j(z) * (vc[j][:] * vs[j])
 *
 * kc [B][*][d_qk] and vc [B][*][d_v] int8 codes with batch strides skc_b, svc_b
 * elements; ks, vs [B][*] fp32 with batch strides sks_b, svs_b. */
void oracle_sparse_attn_i8kv(const uint16_t *q, const int8_t *kc, int64_t skc_b,
                             const float *ks, int64_t sks_b, const int8_t *vc, int64_t svc_b,
                             const float *vs, int64_t svs_b, const int32_t *seq_len,
                             const int32_t *idx, int B, int T, int H_q, int d_qk, int d_v,
                             int P, int k, double scale, uint16_t *out, float *lse)
{
    const int64_t cap = (int64_t)k * P > 0 ? (int64_t)k * P : 1;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)cap);
    double *zs = (double *)malloc(sizeof(double) * (size_t)cap);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d_v);
    for (int b = 0; b < B; ++b) {
        const int64_t n_groups = seq_len[b] / P;
        for (int t = 0; t < T; ++t) {
            const int32_t *chosen = idx + ((int64_t)b * T + t) * k;
            int64_t nt = 0;  /* the tokens of the chosen complete groups */
            for (int s = 0; s < k; ++s) {
                if (chosen[s] < 0 || chosen[s] >= n_groups)
                    continue;
                for (int i = 0; i < P; ++i)
                    rows[nt++] = (int64_t)chosen[s] * P + i;
            }
            for (int h = 0; h < H_q; ++h) {
                const int64_t row = ((int64_t)b * T + t) * H_q + h;
                const uint16_t *qv = q + row * d_qk;
                uint16_t *ov = out + row * d_v;
                if (nt == 0) {
                    for (int i = 0; i < d_v; ++i)
                        ov[i] = 0;
                    if (lse)
                        lse[row] = -INFINITY;
                    continue;
                }
                double zmax = -INFINITY;
                for (int64_t j = 0; j < nt; ++j) {
                    const int8_t *kr = kc + b * skc_b + rows[j] * d_qk;
                    const float kscale = ks[b * sks_b + rows[j]];
                    double qk = 0.0;
                    for (int i = 0; i < d_qk; ++i)
                        qk += bf16_value(qv[i]) * oracle_i8_value(kr[i], kscale);
                    zs[j] = scale * qk;
                    zmax = zs[j] > zmax ? zs[j] : zmax;
                }
                double denom = 0.0;
                for (int i = 0; i < d_v; ++i)
                    acc[i] = 0.0;
                for (int64_t j = 0; j < nt; ++j) {
                    const double wj = exp(zs[j] - zmax);
                    denom += wj;
                    const int8_t *vr = vc + b * svc_b + rows[j] * d_v;
                    const float vscale = vs[b * svs_b + rows[j]];
                    for (int i = 0; i < d_v; ++i)
                        acc[i] += wj * oracle_i8_value(vr[i], vscale);
                }
                for (int i = 0; i < d_v; ++i)
                    ov[i] = oracle_bf16_from_double(acc[i] / denom);
                if (lse)
                    lse[row] = (float)(zmax + log(denom));
            }
        }
    }
    free(acc);
    free(zs);
    free(rows);
}
