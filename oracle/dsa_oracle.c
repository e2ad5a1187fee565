/*
 * dsa_oracle.c -- plain FP64 CPU oracle for the DSA decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see dsa_oracle.h).  Written for a reader who
 * checks it against the pages by eye: no blocking, no fusion, no reordering
 * beyond the definitions below.  Compiled with plain `gcc -O2` (no fast-math).
 */
#include "dsa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32: widen and reinterpret. */
double dsa_oracle_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3: sign, 4-bit exponent (bias 7), 3-bit mantissa.
 * Exponent field 0 is subnormal: m * 2^-3 * 2^(1-7).  S.1111.111 is NaN;
 * there is no infinity. */
double dsa_oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round to nearest, ties to even, saturating.  The non-negative finite codes
 * 0x00..0x7E are increasing in value, so the two neighbours of |v| are found
 * by a scan; "even" is the code whose mantissa LSB is 0. */
uint8_t dsa_oracle_e4m3_encode(double v, int *near_midpoint)
{
    const double max_finite = dsa_oracle_e4m3_value(0x7E); /* 448 */
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (near_midpoint)
        *near_midpoint = 0;
    if (isnan(v))
        return 0x7F;
    if (a >= max_finite)
        return (uint8_t)(sign | 0x7E);
    /* largest code whose value is <= a */
    int lo = 0;
    for (int c = 0; c <= 0x7E; ++c) {
        if (dsa_oracle_e4m3_value((uint8_t)c) <= a)
            lo = c;
        else
            break;
    }
    int hi = lo + 1; /* exists because a < 448 */
    double vlo = dsa_oracle_e4m3_value((uint8_t)lo);
    double vhi = dsa_oracle_e4m3_value((uint8_t)hi);
    double mid = 0.5 * (vlo + vhi);
    int pick;
    if (a < mid)
        pick = lo;
    else if (a > mid)
        pick = hi;
    else
        pick = (lo & 1) ? hi : lo;
    if (near_midpoint && fabs(a - mid) <= ldexp(mid, -20))
        *near_midpoint = 1;
    return (uint8_t)(sign | (uint8_t)pick);
}

/* ------------------------------------------------------------------------ */
/* S0: latent write (vanilla RMSNorm -> scale by fl32(1/kv_scale) -> E4M3)   */
/* glm5next_dsa/layer.rs: module header trap "Two RMSNorm kernels differ     */
/* only by a +1" (GLM takes x * rms * w), decode_k "kv path" (the latent     */
/* write receives eps and 1/kv_scale as f32), and the kv_scale field ("the   */
/* write takes 1/scale").                                                    */
/* ------------------------------------------------------------------------ */
void dsa_oracle_latent_write_row(int dim, const uint16_t *kv_a_row,
                                 const uint16_t *norm_w, float eps, float kv_scale,
                                 uint8_t *out_codes, double *pre, uint8_t *near_mid)
{
    double sum_sq = 0.0;
    for (int i = 0; i < dim; ++i) {
        double x = dsa_oracle_bf16_value(kv_a_row[i]);
        sum_sq += x * x;
    }
    double mean_sq = sum_sq / (double)dim;
    double rms = 1.0 / sqrt(mean_sq + (double)eps);
    float inv_scale = 1.0f / kv_scale; /* the inverse is an FP32 value */
    for (int i = 0; i < dim; ++i) {
        double x = dsa_oracle_bf16_value(kv_a_row[i]);
        double w = dsa_oracle_bf16_value(norm_w[i]);
        double y = x * rms * w;
        double v = y * (double)inv_scale;
        int nm = 0;
        out_codes[i] = dsa_oracle_e4m3_encode(v, &nm);
        if (pre)
            pre[i] = v;
        if (near_mid)
            near_mid[i] = (uint8_t)nm;
    }
}

/* ------------------------------------------------------------------------ */
/* S1: indexer score.  glm5next_dsa/layer.rs module header (q_idx, k_normed, */
/* gate and head weights feed select_tokens; weights_proj already carries    */
/* index_heads^-0.5, the score kernel does not scale), with the per-token    */
/* scalar gate multiplying the head-weighted ReLU sum.                       */
/* ------------------------------------------------------------------------ */
void dsa_oracle_index_scores_row(int heads, int dim, const float *q, const float *w,
                                 const uint16_t *k, const uint16_t *gate,
                                 int64_t n, const int64_t *tokens,
                                 double *s_out, double *a_out, double *m_out)
{
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens ? tokens[i] : i;
        const uint16_t *kt = k + t * (int64_t)dim;
        double g = dsa_oracle_bf16_value(gate[t]);
        double sum = 0.0, sum_abs = 0.0, terms = 0.0;
        for (int h = 0; h < heads; ++h) {
            double dot = 0.0, dot_abs = 0.0;
            for (int d = 0; d < dim; ++d) {
                double term = (double)q[h * dim + d] * dsa_oracle_bf16_value(kt[d]);
                dot += term;
                dot_abs += fabs(term);
            }
            double relu = dot > 0.0 ? dot : 0.0;
            sum += (double)w[h] * relu;
            sum_abs += fabs((double)w[h]) * relu;
            terms += fabs((double)w[h]) * dot_abs;
        }
        s_out[i] = g * sum;
        if (a_out)
            a_out[i] = g * sum_abs;
        if (m_out)
            m_out[i] = g * terms;
    }
}

/* ------------------------------------------------------------------------ */
/* S2: top-k under the total order (score DESC, index ASC).                  */
/* glm5next_dsa/layer.rs, notes on batch_select_enabled and                  */
/* select_rows_batched: the selection is unique because the order is total.  */
/* ------------------------------------------------------------------------ */
typedef struct {
    double score;
    int64_t index;
} scored_token;

static int by_score_desc_index_asc(const void *pa, const void *pb)
{
    const scored_token *a = (const scored_token *)pa;
    const scored_token *b = (const scored_token *)pb;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    if (a->index < b->index)
        return -1;
    if (a->index > b->index)
        return 1;
    return 0;
}

static int by_int32_asc(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

int dsa_oracle_select_topk_row(int64_t len, int topk, const double *scores, int32_t *sel)
{
    int64_t n = len < (int64_t)topk ? len : (int64_t)topk;
    if (n < 0)
        n = 0;
    if (len > 0) {
        scored_token *all = (scored_token *)malloc((size_t)len * sizeof *all);
        for (int64_t t = 0; t < len; ++t) {
            all[t].score = scores[t];
            all[t].index = t;
        }
        qsort(all, (size_t)len, sizeof *all, by_score_desc_index_asc);
        for (int64_t i = 0; i < n; ++i)
            sel[i] = (int32_t)all[i].index;
        free(all);
        qsort(sel, (size_t)n, sizeof *sel, by_int32_asc);
    }
    for (int64_t i = n; i < topk; ++i)
        sel[i] = -1;
    return (int)n;
}

/* ------------------------------------------------------------------------ */
/* S3: absorbed NoPE MLA gather-attend.  glm5next_dsa/layer.rs: module       */
/* header (Q absorbed into the 512-d latent), attend_rows (K and V are the   */
/* same latent pool; each row reads its own selection, seq_len and block-    */
/* table row), decode_k (slot = block * block_size + pos % block_size).      */
/* ------------------------------------------------------------------------ */
static int slot_of(int64_t j, const int32_t *bt, int max_blocks, int block_size,
                   int64_t nslots, int64_t *slot)
{
    int64_t logical = j / block_size;
    if (logical < 0 || logical >= max_blocks)
        return -1;
    int64_t phys = bt[logical];
    if (phys < 0)
        return -1;
    int64_t s = phys * block_size + j % block_size;
    if (s >= nslots)
        return -1;
    *slot = s;
    return 0;
}

int dsa_oracle_mla_decode_row(int heads, int dim, const uint16_t *Q,
                              const uint8_t *pool, int64_t nslots,
                              const int32_t *bt, int max_blocks, int block_size,
                              int64_t seq_len, const int32_t *sel, int topk,
                              float kv_scale, float sm_scale,
                              double *out, double *lse, double *zmag)
{
    /* the selected, dequantised latent rows */
    int n = 0;
    double *khat = (double *)malloc((size_t)(topk > 0 ? topk : 1) * (size_t)dim * sizeof(double));
    for (int i = 0; i < topk; ++i) {
        int64_t j = sel[i];
        int64_t slot;
        if (j == -1)
            continue;
        if (j < 0 || j >= seq_len || slot_of(j, bt, max_blocks, block_size, nslots, &slot)) {
            free(khat);
            return -1;
        }
        for (int c = 0; c < dim; ++c)
            khat[(size_t)n * dim + c] =
                dsa_oracle_e4m3_value(pool[slot * dim + c]) * (double)kv_scale;
        ++n;
    }
    double *z = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    for (int h = 0; h < heads; ++h) {
        double *o = out + (size_t)h * dim;
        for (int c = 0; c < dim; ++c)
            o[c] = 0.0;
        if (n == 0) {
            lse[h] = -INFINITY;
            if (zmag)
                zmag[h] = 0.0;
            continue;
        }
        double m = -INFINITY;
        double mag_max = 0.0;
        for (int j = 0; j < n; ++j) {
            double dot = 0.0, mag = 0.0;
            for (int c = 0; c < dim; ++c) {
                const double term = dsa_oracle_bf16_value(Q[(size_t)h * dim + c]) * khat[(size_t)j * dim + c];
                dot += term;
                mag += fabs(term);
            }
            z[j] = (double)sm_scale * dot;
            if (z[j] > m)
                m = z[j];
            if (fabs((double)sm_scale) * mag > mag_max)
                mag_max = fabs((double)sm_scale) * mag;
        }
        if (zmag)
            zmag[h] = mag_max;
        double denom = 0.0;
        for (int j = 0; j < n; ++j)
            denom += exp(z[j] - m);
        for (int j = 0; j < n; ++j) {
            double p = exp(z[j] - m) / denom;
            for (int c = 0; c < dim; ++c)
                o[c] += p * khat[(size_t)j * dim + c];
        }
        lse[h] = m + log(denom);
    }
    free(z);
    free(khat);
    return 0;
}

int dsa_oracle_dense_mla_row(int heads, int dim, const uint16_t *Q,
                             const uint8_t *pool, int64_t nslots,
                             const int32_t *bt, int max_blocks, int block_size,
                             int64_t seq_len, float kv_scale, float sm_scale,
                             double *out, double *lse)
{
    /* logits[h][t] for every visible token */
    size_t L = (size_t)(seq_len > 0 ? seq_len : 0);
    double *logits = (double *)malloc((L ? L : 1) * (size_t)heads * sizeof(double));
    int64_t *slots = (int64_t *)malloc((L ? L : 1) * sizeof(int64_t));
    for (size_t t = 0; t < L; ++t) {
        if (slot_of((int64_t)t, bt, max_blocks, block_size, nslots, &slots[t])) {
            free(logits);
            free(slots);
            return -1;
        }
    }
    for (int h = 0; h < heads; ++h)
        for (size_t t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int c = 0; c < dim; ++c) {
                double q = dsa_oracle_bf16_value(Q[(size_t)h * dim + c]);
                double kv = dsa_oracle_e4m3_value(pool[slots[t] * dim + c]) * (double)kv_scale;
                acc += q * kv;
            }
            logits[(size_t)h * L + t] = acc * (double)sm_scale;
        }
    for (int h = 0; h < heads; ++h) {
        double *row = logits + (size_t)h * L;
        double mx = -INFINITY, total = 0.0;
        for (size_t t = 0; t < L; ++t)
            mx = row[t] > mx ? row[t] : mx;
        for (size_t t = 0; t < L; ++t)
            total += exp(row[t] - mx);
        lse[h] = L ? mx + log(total) : -INFINITY;
        for (int c = 0; c < dim; ++c) {
            double acc = 0.0;
            for (size_t t = 0; t < L; ++t) {
                double kv = dsa_oracle_e4m3_value(pool[slots[t] * dim + c]) * (double)kv_scale;
                acc += exp(row[t] - mx) / total * kv;
            }
            out[(size_t)h * dim + c] = acc;
        }
    }
    free(logits);
    free(slots);
    return 0;
}

int64_t dsa_oracle_bt_entries_needed(int64_t seq_len, int64_t k, int64_t block_size)
{
    int64_t bs = block_size > 0 ? block_size : 1;
    return (seq_len + k) / bs + 2;
}

/* ------------------------------------------------------------------------ */
/* Batched projection (the K-token verify's weight sweep)                    */
/* ------------------------------------------------------------------------ */

/* "glm5next_dsa/layer.rs", the gemm helper (C[M, N] = A[M, K] @ B[N, K]^T)
 * and the notes on decode_k / dense_gemv_bf16_batchm: K rows of one sequence
 * multiply the same weight, each row exactly as a single-row call would.
 * One row of A against every row of B, accumulated in double in k order. */
void dsa_oracle_dense_mm_row(int n, int k, const uint16_t *a_row, const uint16_t *b,
                             double *c, double *mag)
{
    for (int j = 0; j < n; ++j) {
        double acc = 0.0, m = 0.0;
        for (int i = 0; i < k; ++i) {
            double prod = dsa_oracle_bf16_value(a_row[i]) *
                          dsa_oracle_bf16_value(b[(int64_t)j * k + i]);
            acc += prod;
            m += fabs(prod);
        }
        c[j] = acc;
        if (mag)
            mag[j] = m;
    }
}

/* ------------------------------------------------------------------------ */
/* Indexer write side: k_norm                                                */
/* ------------------------------------------------------------------------ */

/* "glm5next_dsa/layer.rs", module header trap 2 and indexer_forward: the
 * indexer's k_norm is an nn.LayerNorm with a bias (mean subtraction, the
 * biased variance, weight and bias), applied to the wk projection of the
 * token before it is stored in the key cache. */
void dsa_oracle_layer_norm_row(int dim, const uint16_t *x, const uint16_t *w, const uint16_t *b,
                               float eps, double *y, double *mag)
{
    double mu = 0.0, var = 0.0;
    for (int d = 0; d < dim; ++d)
        mu += dsa_oracle_bf16_value(x[d]);
    mu /= dim;
    for (int d = 0; d < dim; ++d) {
        double c = dsa_oracle_bf16_value(x[d]) - mu;
        var += c * c;
    }
    var /= dim;
    double inv = 1.0 / sqrt(var + (double)eps);
    for (int d = 0; d < dim; ++d) {
        double t = (dsa_oracle_bf16_value(x[d]) - mu) * inv * dsa_oracle_bf16_value(w[d]);
        y[d] = t + dsa_oracle_bf16_value(b[d]);
        if (mag)
            mag[d] = fabs(t) + fabs(dsa_oracle_bf16_value(b[d]));
    }
}

/* ------------------------------------------------------------------------ */
/* Pool-compressed selection, the half the pages specify.                   */
/* "glm5next_dsa/layer.rs", the notes above batch_select_enabled and on      */
/* select_rows_batched: a pool is a candidate for row r only when it is      */
/* complete (pool_valid) and its last token is visible to the row            */
/* (end <= q_pos[r]); non-candidates score -FLT_MAX and are left out; the    */
/* pools are taken under the total order (score DESC, then pool index ASC);  */
/* the per-row count row_select_k = min(select_k, (q_pos[r] + 1) / KP) sets  */
/* both the number of pools taken and the base of the visible tail, which   */
/* dsa_expand_selection writes after the pools' tokens.  How the pool scores */
/* are computed (the gate and ape compression) is not on the pages; the      */
/* caller supplies them.                                                     */
/* ------------------------------------------------------------------------ */
static int64_t row_select_k(int select_k, int kp, int64_t q_pos)
{
    int64_t visible = q_pos + 1 >= 0 ? (q_pos + 1) / (kp > 0 ? kp : 1) : 0;
    return visible < (int64_t)select_k ? visible : (int64_t)select_k;
}

int dsa_oracle_select_pools_row(int64_t npools, const float *scores, const uint8_t *valid,
                                int64_t q_pos, int kp, int select_k, int32_t *sel)
{
    int64_t want = row_select_k(select_k, kp, q_pos);
    /* candidates of this row, then the total order over them */
    scored_token *cand = (scored_token *)malloc((size_t)(npools > 0 ? npools : 1) * sizeof *cand);
    int64_t nc = 0;
    for (int64_t p = 0; p < npools; ++p) {
        int64_t end = (p + 1) * (int64_t)kp - 1;
        if (valid[p] && end <= q_pos) {
            cand[nc].score = (double)scores[p];
            cand[nc].index = p;
            ++nc;
        }
    }
    qsort(cand, (size_t)nc, sizeof *cand, by_score_desc_index_asc);
    int64_t n = nc < want ? nc : want;
    for (int64_t i = 0; i < n; ++i)
        sel[i] = (int32_t)cand[i].index;
    for (int64_t i = n; i < select_k; ++i)
        sel[i] = -1;
    free(cand);
    return (int)n;
}

void dsa_oracle_expand_selection_row(int select_k, int kp, const int32_t *pools, int64_t q_pos,
                                     int out_width, int32_t *tokens)
{
    int64_t k = row_select_k(select_k, kp, q_pos);
    for (int i = 0; i < out_width; ++i)
        tokens[i] = -1;
    /* the selected pools' tokens, pool i at [i*KP, (i+1)*KP) */
    for (int64_t i = 0; i < k; ++i)
        if (pools[i] >= 0)
            for (int j = 0; j < kp; ++j)
                if (i * kp + j < out_width)
                    tokens[i * kp + j] = (int32_t)((int64_t)pools[i] * kp + j);
    /* the visible tail: the tokens after the last complete pool, up to q_pos */
    int64_t tail_start = q_pos + 1 >= 0 ? ((q_pos + 1) / kp) * kp : 0;
    for (int64_t t = tail_start; t <= q_pos; ++t) {
        int64_t at = k * kp + (t - tail_start);
        if (at < out_width)
            tokens[at] = (int32_t)t;
    }
}
