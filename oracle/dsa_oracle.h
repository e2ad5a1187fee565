/*
 * dsa_oracle.h -- plain, slow, FP64 CPU oracle for the DSA decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code; it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can say what the right answer is.  It shares
 * no source with the CUDA library.
 *
 * What it follows (pages of the spark_model documentation):
 *   - "glm5next_dsa/layer.rs" source page, module header ("Decode, end to end"
 *     diagram and the four silent-wrong-answer traps), decode_k ("kv path:
 *     latent -> FP8 -> paged slot"), attend_rows, and the selection notes on
 *     batch_select_enabled / select_rows_batched (total order score DESC,
 *     index ASC).
 *   - "Struct Glm5NextDsaLayer" rustdoc page, field kv_scale ("the write takes
 *     1/scale").
 * Number formats are written from their published definitions:
 *   - bfloat16: the upper 16 bits of an IEEE-754 binary32.
 *   - FP8 E4M3 (OCP 8-bit floating point spec): 1 sign, 4 exponent bits with
 *     bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, max 448.
 *
 * Every function works on one decode row (or one latent row) at a time; the
 * caller loops over rows.  All accumulation is in double.
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact value of a bfloat16 bit pattern. */
double dsa_oracle_bf16_value(uint16_t bits);

/* Exact value of an FP8 E4M3 code (NaN for 0x7F / 0xFF). */
double dsa_oracle_e4m3_value(uint8_t code);

/* Round-to-nearest-even, saturating to +-448, of a real value to E4M3.
 * NaN in -> 0x7F.  The sign of zero follows the sign of the input.
 * If near_midpoint is non-NULL it is set to 1 when |v| lies within a relative
 * distance 2^-20 of a rounding midpoint (a value two adjacent codes are
 * equally near), else 0. */
uint8_t dsa_oracle_e4m3_encode(double v, int *near_midpoint);

/* S0 -- latent write for one row.
 *   y_i = x_i / sqrt(mean_j(x_j^2) + eps) * w_i   (vanilla RMSNorm: w, not 1+w)
 *   v_i = y_i * fl32(1/kv_scale)                  (the inverse taken in FP32)
 *   out_i = E4M3_RNE_satfinite(v_i)
 * kv_a_row, norm_w: [dim] bf16 bits.  out_codes: [dim] codes.  pre (optional):
 * [dim] values before rounding.  near_mid (optional): [dim] midpoint flags. */
void dsa_oracle_latent_write_row(int dim, const uint16_t *kv_a_row,
                                 const uint16_t *norm_w, float eps, float kv_scale,
                                 uint8_t *out_codes, double *pre, uint8_t *near_mid);

/* S1 -- lightning-indexer score of one query row at n tokens.
 *   a_h(t) = sum_d q[h][d] * k[t][d]
 *   s(t)   = gate[t] * sum_h w[h] * max(a_h(t), 0)
 *   A(t)   = gate[t] * sum_h |w[h]| * max(a_h(t), 0)   (magnitude scale for tolerances)
 *   M(t)   = gate[t] * sum_h |w[h]| * sum_d |q[h][d] * k[t][d]|
 *            (size of the terms summed: the conditioning scale of s(t))
 * q: [heads][dim] float; w: [heads] float (already carrying heads^-0.5);
 * k: [*][dim] bf16 bits for this row's sequence (token t at k + t*dim);
 * gate: [*] bf16 bits.  tokens: the n token indices to score, or NULL for
 * tokens 0..n-1.  s_out: [n]; a_out, m_out (optional): [n]. */
void dsa_oracle_index_scores_row(int heads, int dim, const float *q, const float *w,
                                 const uint16_t *k, const uint16_t *gate,
                                 int64_t n, const int64_t *tokens,
                                 double *s_out, double *a_out, double *m_out);

/* S2 -- top-k of one row.  Orders tokens 0..len-1 by (score DESC, index ASC),
 * keeps the first min(topk, len), writes them to sel[0..] in ASCENDING index
 * order and fills sel[n..topk) with -1.  Returns n.  Scores must not be NaN. */
int dsa_oracle_select_topk_row(int64_t len, int topk, const double *scores, int32_t *sel);

/* S3 -- absorbed, NoPE MLA gather-attend of one row over its selection.
 * Q: [heads][dim] bf16 bits (latent space).  pool: [nslots][dim] E4M3 codes.
 * bt: this row's block table, [max_blocks] ids.  A selected token j maps to
 * slot bt[j / block_size] * block_size + j % block_size.
 *   Khat_j  = e4m3(pool[slot_j]) * kv_scale        (K = V = latent)
 *   z_hj    = sm_scale * sum_c Q[h][c] * Khat_j[c]
 *   p_hj    = softmax_j(z_hj) over the selected j only
 *   out[h]  = sum_j p_hj * Khat_j ;  lse[h] = log sum_j exp(z_hj)
 * Entries of sel equal to -1 are padding and are skipped.  With nothing
 * selected, out = 0 and lse = -inf.  zmag (optional): [heads], the largest
 * over the selected j of |sm_scale| * sum_c |Q[h][c] * Khat_j[c]|, the size of
 * the terms a logit sums (the conditioning scale of z and lse; 0 when nothing
 * is selected).  Returns 0, or -1 if an entry is outside [0, seq_len), or
 * maps outside the table or the pool. */
int dsa_oracle_mla_decode_row(int heads, int dim, const uint16_t *Q,
                              const uint8_t *pool, int64_t nslots,
                              const int32_t *bt, int max_blocks, int block_size,
                              int64_t seq_len, const int32_t *sel, int topk,
                              float kv_scale, float sm_scale,
                              double *out, double *lse, double *zmag);

/* Dense MLA attention of one row over every token 0..seq_len-1, written
 * independently of the gather path (a full logits matrix, then a two-pass
 * softmax).  Used only to pin the gather path: with topk >= seq_len the two
 * must agree.  Same arguments and results as the gather form. */
int dsa_oracle_dense_mla_row(int heads, int dim, const uint16_t *Q,
                             const uint8_t *pool, int64_t nslots,
                             const int32_t *bt, int max_blocks, int block_size,
                             int64_t seq_len, float kv_scale, float sm_scale,
                             double *out, double *lse);

/* Block-table entries the paged gather can index for k query rows starting at
 * seq_len, plus one entry of slack (glm5next_dsa/layer.rs, bt_entries_needed:
 * the gather touches block_table[pos / block_size] for pos in [0, seq_len+k)).
 * A block size of 0 is treated as 1. */
int64_t dsa_oracle_bt_entries_needed(int64_t seq_len, int64_t k, int64_t block_size);

/* Batched projection, one row of A:
 *   c[j]   = sum_i a_row[i] * b[j][i]       (a_row: [k] bf16, b: [n][k] bf16)
 *   mag[j] = sum_i |a_row[i] * b[j][i]|     (optional; scale for tolerances)
 * in double, i ascending. */
void dsa_oracle_dense_mm_row(int n, int k, const uint16_t *a_row, const uint16_t *b,
                             double *c, double *mag);

/* Indexer k_norm (nn.LayerNorm with a bias) of one row:
 *   mu = sum_d x_d / dim,  var = sum_d (x_d - mu)^2 / dim
 *   y_d = (x_d - mu) / sqrt(var + eps) * w_d + b_d
 * x, w, b: [dim] bf16 bits; y: [dim]; mag (optional): [dim]
 * |(x_d - mu) / sqrt(var + eps) * w_d| + |b_d| (scale for tolerances). */
void dsa_oracle_layer_norm_row(int dim, const uint16_t *x, const uint16_t *w, const uint16_t *b,
                               float eps, double *y, double *mag);

/* Pool-compressed selection of one row (the part the pages specify; the pool
 * scores themselves are the caller's).  Pool p covers tokens [p*kp, (p+1)*kp)
 * and is a candidate iff valid[p] != 0 and (p+1)*kp - 1 <= q_pos.  With
 * row_select_k = min(select_k, (q_pos+1) / kp), the first min(row_select_k,
 * #candidates) candidates under (score DESC, pool index ASC) are written to
 * sel[0..) in that order; the rest of sel[0..select_k) is -1.  Returns the
 * number written.  scores, valid: [npools]. */
int dsa_oracle_select_pools_row(int64_t npools, const float *scores, const uint8_t *valid,
                                int64_t q_pos, int kp, int select_k, int32_t *sel);

/* Expansion of one row's pool selection to tokens: for i < row_select_k,
 * tokens[i*kp + j] = pools[i]*kp + j (j < kp; -1 where pools[i] is -1), then
 * the visible tail -- tokens floor((q_pos+1)/kp)*kp .. q_pos -- from index
 * row_select_k*kp on; every other entry of tokens[0..out_width) is -1. */
void dsa_oracle_expand_selection_row(int select_k, int kp, const int32_t *pools, int64_t q_pos,
                                     int out_width, int32_t *tokens);

#ifdef __cplusplus
}
#endif

#endif /* DSA_ORACLE_H */
