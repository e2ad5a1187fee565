/*
 * dsa.h -- C ABI of libdsa_gb300: the DSA decode hot path of the GLM-5.3
 * sparse layers on one GB300 (sm_103a).
 *
 * Per decode row the path is
 *   S0 dsa_latent_write    RMSNorm + FP8 quantisation + paged slot write of the
 *                          row's new latent
 *   S1 dsa_index_scores    lightning-indexer score of every visible token
 *   S2 dsa_select_topk     per-row top-k of those scores
 *   S3 dsa_mla_decode_fp8  absorbed NoPE MLA gather-attend over the selection
 * issued in that order on one stream.  Around the path, for the K-token
 * verify and the indexer's write side:
 *      dsa_dense_mm_bf16   batched projection: up to 16 rows per sweep of a
 *                          bf16 weight, each row bit-identical to a one-row call
 *      dsa_indexer_write   the indexer key's LayerNorm (with bias) and its store
 *                          at the row's device-side arena position
 * and the pool-compressed form of the selection (over caller-supplied pool
 * scores):
 *      dsa_select_pools    top pools per row under (score DESC, pool ASC)
 *      dsa_expand_selection  pools to tokens, plus the visible tail
 * Sources (spark_model documentation):
 * the "glm5next_dsa/layer.rs" source page (module header: decode data flow
 * and its traps; decode_k: latent write, per-row metadata, one attend for all
 * rows; attend_rows; the selection notes on a total order) and the "Struct
 * Glm5NextDsaLayer" rustdoc page (kv_scale, decode_k).
 *
 * Conventions for every entry point
 *   - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *     owned by the caller and unchanged until the work on `stream` completes.
 *     The library never allocates, frees, copies host<->device or
 *     synchronises inside these calls (so the calls can be recorded into a
 *     CUDA graph by the caller).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous: a DSA_OK return means the work was enqueued.
 *   - bf16 tensors are passed as uint16_t bit patterns; FP8 as uint8_t E4M3
 *     codes (OCP: bias 7, max 448, no infinities).
 *   - Argument errors detectable on the host return DSA_ERR_INVALID_ARG or
 *     DSA_ERR_UNSUPPORTED before anything is launched.  Launch failures return
 *     DSA_ERR_CUDA.  Values only visible on the device (a seq_len above
 *     max_len, a selected index outside [0, seq_len), a negative block id, a
 *     slot outside the pool, mismatched arena bases) make the kernel skip the
 *     offending access and record the first such error in a sticky device
 *     error word that dsa_get_error() reads; kernels never trap.  Every wait
 *     inside a kernel is bounded and records DSA_DEVERR_TIMEOUT when it gives
 *     up.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 4
#define DSA_LATENT_DIM 512

typedef enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,
    DSA_ERR_UNSUPPORTED = 2,
    DSA_ERR_CUDA = 3,
    DSA_ERR_DEVICE = 4,      /* dsa_get_error found a recorded device-side error */
    DSA_ERR_WORKSPACE = 5    /* workspace missing or smaller than dsa_workspace_bytes() */
} dsa_status;

/* Codes recorded in the device error word. */
enum {
    DSA_DEVERR_NONE = 0,
    DSA_DEVERR_SEQ_LEN = 1,   /* seq_len < 0 or > max_len                               */
    DSA_DEVERR_SLOT = 2,      /* latent-write slot outside [0, nslots)                  */
    DSA_DEVERR_SELECT = 3,    /* selected index outside [0, seq_len) and not -1         */
    DSA_DEVERR_BLOCK = 4,     /* block-table entry missing, negative or past the pool   */
    DSA_DEVERR_ARENA = 5,     /* idx_base invalid, or rows of one group differ in base  */
    DSA_DEVERR_POSITION = 6,  /* positions[r] != seq_lens[r]-1, or slot != table slot   */
    DSA_DEVERR_TIMEOUT = 7,   /* a bounded wait inside a kernel gave up                 */
    DSA_DEVERR_BEHIND = 8     /* a sequence's indexer keys stop short of its length:
                                 rows were never written (lockstep with the KV cache)  */
};

/*
 * Per-row metadata of one call ("glm5next_dsa/layer.rs", decode_k: the K-row
 * attn_metadata -- positions [k] u32, slot [k] i64, seq_len [k] i32,
 * block_table [k][max_blocks_per_seq] i32 -- at stable device addresses; row r
 * reads element r of each).  All pointers are device pointers.
 */
typedef struct dsa_rows {
    const uint32_t *positions;  /* [rows] token position of the row (= seq_len-1); may be
                                   NULL.  When given, dsa_latent_write checks it against
                                   seq_lens and the table and refuses inconsistent rows. */
    const int64_t *slots;       /* [rows] paged slot of the row's new latent:
                                   block_table[pos/block_size]*block_size + pos%block_size.
                                   Read only by dsa_latent_write; may be NULL otherwise.  */
    const int32_t *seq_lens;    /* [rows] the row sees tokens [0, seq_len)               */
    const int32_t *block_table; /* row r at block_table + r*bt_stride, max_blocks_per_seq
                                   entries of physical block ids; -1 = none.             */
    int32_t max_blocks_per_seq; /* entries per table row (bounds every lookup)           */
    int32_t bt_stride;          /* elements between table rows; 0 = every row uses row 0
                                   (rows of one sequence sharing one table)              */
    int32_t block_size;         /* tokens per paged block, > 0                           */
    int32_t rows;               /* R >= 1                                                */
} dsa_rows;

/*
 * S0 -- latent write ("glm5next_dsa/layer.rs", module header trap 1 and
 * decode_k "kv path: latent -> FP8 -> paged slot"; "Struct Glm5NextDsaLayer",
 * kv_scale: the write takes 1/scale).  For each row r:
 *   y = kv_a[r] * rsqrt(mean(kv_a[r]^2) + eps) * norm_w      (vanilla: w, not 1+w)
 *   pool[slots[r]][i] = E4M3_RNE_satfinite(y[i] * fl32(1/kv_scale))
 * The norm and scaling are computed in double, with one rounding to FP8.
 *   kv_a    [rows][latent_dim] bf16      norm_w [latent_dim] bf16
 *   pool    [nslots][latent_dim] FP8, written in place at the rows' slots
 * latent_dim must be 512.  A slot outside [0, nslots) (or a row inconsistent
 * with `positions`, when given) is skipped and recorded on the device.
 */
dsa_status dsa_latent_write(const dsa_rows *rows, const uint16_t *kv_a, const uint16_t *norm_w,
                            uint8_t *pool, int64_t nslots, int32_t latent_dim, float eps,
                            float kv_scale, void *stream);

/*
 * S1 -- lightning-indexer scores ("glm5next_dsa/layer.rs", module header:
 * q_idx, k_normed, gate and the head weights feed select_tokens; trap 3:
 * weights_proj already carries index_heads^-0.5 and the score does not scale).
 * For each row r and token t in [0, seq_lens[r]):
 *   scores[r*max_len + t] = gate[b+t] * sum_h head_w[r][h] * max(0, sum_d q_idx[r][h][d]*idx_k[b+t][d])
 * with b = idx_base[r].  Entries t >= seq_lens[r] of a scores row are not written.
 *   q_idx  [rows][index_heads][index_dim] fp32   head_w [rows][index_heads] fp32
 *   idx_k  [idx_tokens][index_dim] bf16 (key arena, all sequences)
 *   idx_gate [idx_tokens] bf16 (per-token scalar gate)
 *   idx_base [rows] int64: the row's sequence start in the arena
 *   scores [rows][max_len] fp32 (output)
 * rows_per_seq: consecutive rows that share one sequence (a K-token verify);
 * they must have equal idx_base (checked on the device) and share each key
 * tile they read, up to 64 score columns (rows x index_heads) per read.
 * rows must be a multiple of rows_per_seq.
 * idx_written (optional, may be NULL): [rows / rows_per_seq] int32, the rows
 * of each sequence's keys written so far (as kept by dsa_indexer_write); a
 * row whose seq_len exceeds its sequence's count is skipped (scores not
 * written) and recorded as DSA_DEVERR_BEHIND.
 * Supported: index_dim in {64, 128}; index_heads in [1, 256]; idx_k 16-byte
 * aligned; idx_tokens < 2^31.  Each row's result does not depend on
 * rows_per_seq or on the other rows (bit for bit).
 */
dsa_status dsa_index_scores(const dsa_rows *rows, const float *q_idx, const float *head_w,
                            const uint16_t *idx_k, const uint16_t *idx_gate, int64_t idx_tokens,
                            const int64_t *idx_base, int32_t index_heads, int32_t index_dim,
                            int32_t rows_per_seq, int32_t max_len, float *scores,
                            const int32_t *idx_written, void *stream);

/*
 * S1 with flags.  dsa_index_scores is this call with flags 0.
 * DSA_INDEX_INPUTS_BEFORE_PREDECESSOR: the caller asserts that every input of
 * the call (q_idx, head_w, idx_k, idx_gate, idx_base, idx_written and the
 * rows' seq_lens) was complete before the kernel issued just before this call
 * on the stream started -- for instance a decode step whose queries and keys
 * were produced before its latent write, or steps replayed back to back over
 * resident inputs.  The indexer may then load its inputs, run its MMAs and
 * compute its scores while that kernel still runs; its stores to `scores`
 * (which a kernel before may still read) and its completion still wait for
 * that kernel.  Do not set it when the kernel before writes an input (an
 * indexer write or a projection producing q_idx).  The results are
 * bit-identical either way.  Unknown flag bits: DSA_ERR_INVALID_ARG.
 */
#define DSA_INDEX_INPUTS_BEFORE_PREDECESSOR 1u
dsa_status dsa_index_scores_ex(const dsa_rows *rows, const float *q_idx, const float *head_w,
                               const uint16_t *idx_k, const uint16_t *idx_gate, int64_t idx_tokens,
                               const int64_t *idx_base, int32_t index_heads, int32_t index_dim,
                               int32_t rows_per_seq, int32_t max_len, float *scores,
                               const int32_t *idx_written, uint32_t flags, void *stream);

/*
 * S2 -- per-row top-k ("glm5next_dsa/layer.rs", notes on batch_select_enabled
 * and select_rows_batched: the selection is taken under the total order score
 * DESC, then index ASC, so it is unique).  For each row r, the n = min(topk,
 * seq_lens[r]) tokens of [0, seq_lens[r]) that come first under that order are
 * written to sel[r*topk + 0 .. n) in ASCENDING token order; sel[r*topk + n ..
 * topk) = -1.  -0.0 and +0.0 compare equal.  Scores must not be NaN.
 *   scores [rows][max_len] fp32 (as written by dsa_index_scores)
 *   sel    [rows][topk] int32 (output)
 * topk in [1, 65536]; max_len up to about 390k tokens (a row is held in
 * shared memory by a cluster of up to 8 CTAs).  No workspace.
 */
dsa_status dsa_select_topk(const dsa_rows *rows, const float *scores, int32_t max_len,
                           int32_t topk, int32_t *sel, void *stream);

/*
 * S3 -- absorbed NoPE MLA gather-attend over the selection
 * ("glm5next_dsa/layer.rs", module header trap 4: Q arrives absorbed into the
 * 512-d latent space; attend_rows: one launch for all rows, each with its own
 * selection row, seq_len and table row, K and V the same latent pool; decode_k:
 * slot = block*block_size + pos%block_size).  For each row r and head h, over
 * the entries j of sel[r] that are not -1:
 *   Khat_j = e4m3(pool[slot(j)]) * kv_scale
 *   z_j    = sm_scale * (q[r][h] . Khat_j)
 *   out[r][h] = sum_j softmax(z)_j * Khat_j           (bf16, latent space)
 *   lse[r][h] = log sum_j exp(z_j)                     (fp32, optional)
 * A row with nothing selected gets out = 0 and lse = -inf.
 *   q   [rows][heads][latent_dim] bf16       pool [nslots][latent_dim] FP8
 *   sel [rows][topk] int32                   out  [rows][heads][latent_dim] bf16
 * out may also be page-locked host memory mapped into the device's address
 * space (cudaHostAlloc memory under unified addressing): the kernels store the
 * result there directly, with no separate device-to-host copy.
 * latent_dim must be 512; heads a multiple of 16; nslots below 2^31
 * (DSA_ERR_UNSUPPORTED otherwise).  Numerics: q enters the tensor cores as
 * two E4M3 terms per element (hi and the residual, scaled by a power of two
 * per head), which hold a bf16 q exactly except elements more than 2^10
 * below the head's largest |q|, whose last bits fall into E4M3 subnormals;
 * their products with the E4M3 latent accumulate in FP32; the softmax weights enter the weighted sum as two E4M3 terms
 * (about bf16 precision; weights 2^18 below a head's largest drop out), the
 * normalising sums and lse use the unrounded weights.  A row's selection is
 * cut into splits of at most 256 entries (2048 with more than 64 heads; 512
 * with DSA_DECODE_LONG_SPLITS, below) whose count depends only on topk, heads
 * and that flag, so each row's result is bit-identical whatever the other
 * rows of the call are.  With more than one split each
 * split's normalised partial output O/l (a convex combination of latent
 * values, kept in fp16: 2^-11 relative) and its (max, sum) pass through the
 * workspace (L2-resident, discarded after the merge), which must hold
 * dsa_workspace_bytes(rows, heads, topk) bytes, 256-byte aligned
 * (DSA_ERR_WORKSPACE otherwise).
 */
dsa_status dsa_mla_decode_fp8(const dsa_rows *rows, const uint16_t *q, const uint8_t *pool,
                              int64_t nslots, const int32_t *sel, int32_t topk, int32_t heads,
                              int32_t latent_dim, float kv_scale, float sm_scale, uint16_t *out,
                              float *lse_or_null, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * S3 with flags.  dsa_mla_decode_fp8 is this call with flags 0.
 * DSA_DECODE_LONG_SPLITS: with at most 64 heads, splits of at most 512
 * entries instead of 256 (half the CTAs, each twice as long: for launches
 * with many rows, whose CTAs otherwise fill the GPU in more waves; a single
 * row runs faster without it).  The split count then depends on topk, heads
 * and this flag, still never on the other rows: calls whose results must
 * agree bit for bit (a K-row verify and the same rows run one at a time) use
 * the same value of the flag.  The workspace from dsa_workspace_bytes covers
 * both plans.
 * DSA_DECODE_Q_BEFORE_PREDECESSOR: the caller asserts that q was complete
 * before the kernel issued just before this call on the stream started (the
 * usual decode order: q comes from a projection before the indexer, and the
 * kernel before the attend is dsa_select_topk, which writes only sel).  The
 * attend may then load and convert q while that kernel still runs; sel, and
 * everything else a predecessor may write, is still read after the
 * dependency wait.  Without the flag q is read after the wait too.  The
 * results are bit-identical either way.  Unknown flag bits:
 * DSA_ERR_INVALID_ARG.
 */
#define DSA_DECODE_Q_BEFORE_PREDECESSOR 1u
#define DSA_DECODE_LONG_SPLITS 2u
dsa_status dsa_mla_decode_fp8_ex(const dsa_rows *rows, const uint16_t *q, const uint8_t *pool,
                                 int64_t nslots, const int32_t *sel, int32_t topk, int32_t heads,
                                 int32_t latent_dim, float kv_scale, float sm_scale, uint16_t *out,
                                 float *lse_or_null, void *workspace, size_t workspace_bytes,
                                 uint32_t flags, void *stream);

/*
 * S3 for callers that cannot allocate device memory at the point where they
 * run the attend: code that must not take cudaMalloc's implicit device
 * synchronisation on a latency-bound decode path, and code whose device
 * memory belongs to an allocator it may not call (an embedding runtime or a
 * host framework that owns every allocation).  No counterpart on the pages:
 * it is dsa_mla_decode_fp8 with the split partials kept in a device array
 * inside the library instead of a caller workspace.  It allocates nothing and
 * calls no allocating routine.
 *   - Limit: dsa_noalloc_scratch_bytes(rows, heads, topk) must not exceed
 *     DSA_NOALLOC_SCRATCH_BYTES (32 MiB), else DSA_ERR_UNSUPPORTED and
 *     nothing is launched.  Every GPU that loads the library holds that
 *     array until the process exits.
 *   - Set-up: the first call on a device looks the array's device address up
 *     (once per device, with that device current) and keeps it for the life
 *     of the process; make that first call before any stream capture.  The
 *     address belongs to the device's primary context: after
 *     cudaDeviceReset, or under another context on the same device, it is
 *     stale and this entry point must not be used.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls whose work overlaps on
 *     the GPU (other streams, other threads) race on it: serialise them.
 * Other arguments, results and errors are those of dsa_mla_decode_fp8, and
 * the results are bit-identical to that entry point's.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (32u << 20)
dsa_status dsa_mla_decode_fp8_noalloc(const dsa_rows *rows, const uint16_t *q, const uint8_t *pool,
                                      int64_t nslots, const int32_t *sel, int32_t topk,
                                      int32_t heads, int32_t latent_dim, float kv_scale,
                                      float sm_scale, uint16_t *out, float *lse_or_null,
                                      void *stream);

/* Bytes of the library's array that dsa_mla_decode_fp8_noalloc needs for a
 * call of this shape (0 on bad arguments). */
size_t dsa_noalloc_scratch_bytes(int32_t rows, int32_t heads, int32_t topk);

/* Device bytes of the caller-owned workspace that dsa_mla_decode_fp8 needs
 * for a call of this shape (the gather-attend's split partials; 0 when no
 * workspace is needed or on bad arguments). */
size_t dsa_workspace_bytes(int32_t rows, int32_t heads, int32_t topk);

/*
 * Pool-compressed selection, the part the pages specify
 * ("glm5next_dsa/layer.rs", the notes above batch_select_enabled and on
 * select_rows_batched).  Tokens are grouped into pools of kp; pool p holds
 * tokens [p*kp, (p+1)*kp).  For each row r, with q_pos = positions[r]:
 *   - pool p is a candidate iff pool_valid[r*valid_stride + p] != 0 (the pool
 *     is complete) and (p+1)*kp - 1 <= q_pos (its last token is visible);
 *   - row_select_k = min(select_k, (q_pos + 1) / kp);
 *   - sel_pools[r*select_k + i], i < min(row_select_k, #candidates), are the
 *     candidates in the total order (score DESC, then pool index ASC); every
 *     other entry is -1 (a non-candidate is never selected).
 * -0.0 and +0.0 compare equal; scores must not be NaN.  Only pools below
 * (q_pos+1)/kp are read, so a row's result does not depend on max_pools or
 * on the other rows.  How the pool scores are made (the pages' gate [D] and
 * ape [kp][D] compression of the pool's keys) is not on the pages: the caller
 * supplies them.
 *   pool_scores [rows][max_pools] fp32          pool_valid [rows or 1][...] u8
 *   valid_stride: elements between rows of pool_valid, 0 = one shared row
 *   sel_pools   [rows][select_k] int32 (output)
 * rows->positions is required.  kp, select_k >= 1; max_pools in
 * [1, DSA_MAX_POOLS] (DSA_ERR_UNSUPPORTED above).
 */
#define DSA_MAX_POOLS 16384
dsa_status dsa_select_pools(const dsa_rows *rows, const float *pool_scores, int32_t max_pools,
                            const uint8_t *pool_valid, int32_t valid_stride, int32_t kp,
                            int32_t select_k, int32_t *sel_pools, void *stream);

/*
 * Expansion of a pool selection to token indices (same source: the
 * expansion writes the pools' tokens, then the visible tail at
 * row_select_k * kp; the per-row row_select_k applies to both).  For each row
 * r, with q_pos = positions[r] and row_select_k as above:
 *   sel_tokens[r*out_width + i*kp + j] = sel_pools[r*select_k + i]*kp + j
 *       for i < row_select_k, j < kp (-1 where the pool entry is -1);
 *   then the tokens floor((q_pos+1)/kp)*kp .. q_pos (the part of the
 *   incomplete pool the row sees) from entry row_select_k*kp on;
 *   every other entry of the row is -1.
 * The result is a selection row for dsa_mla_decode_fp8 (which skips -1).
 * out_width >= select_k*kp + kp - 1 (room for the longest tail), else
 * DSA_ERR_INVALID_ARG.  rows->positions is required.
 */
dsa_status dsa_expand_selection(const dsa_rows *rows, const int32_t *sel_pools, int32_t kp,
                                int32_t select_k, int32_t *sel_tokens, int32_t out_width,
                                void *stream);

/*
 * Indexer write side for each row's new token ("glm5next_dsa/layer.rs",
 * module header trap 2: indexer.k_norm is an nn.LayerNorm with a bias;
 * indexer_forward: the wk projection of the token lands in the key cache row,
 * normalised in place, the row placed from a DEVICE-side position so that a
 * captured graph replays at the next position).  For each row r, at arena
 * row t = idx_base[r] + positions[r]:
 *   mu = mean_d k_raw[r][d],   var = mean_d (k_raw[r][d] - mu)^2
 *   idx_k[t][d] = bf16_rne((k_raw[r][d] - mu) / sqrt(var + eps) * ln_w[d] + ln_b[d])
 *   idx_gate[t] = gate[r]                                (when gate != NULL)
 *   k_raw [rows][index_dim] bf16 (the wk projection, e.g. from
 *         dsa_dense_mm_bf16), 8-byte aligned
 *   ln_w, ln_b [index_dim] bf16     gate [rows] bf16 or NULL
 *   idx_k [idx_tokens][index_dim] bf16, 8-byte aligned; idx_gate [idx_tokens]
 * rows->positions is required (the new token of row r is position
 * seq_lens[r]-1).  index_dim 64 or 128 (DSA_ERR_UNSUPPORTED otherwise).
 * Numerics: mean, variance and the affine map in double, one rounding to
 * bf16 (nearest, ties to even).  A row whose position is not seq_lens[r]-1
 * (DSA_DEVERR_POSITION) or whose arena row lies outside [0, idx_tokens)
 * (DSA_DEVERR_ARENA) is skipped and recorded.
 * Lockstep with the KV cache ("glm5next_dsa/layer.rs", decode_k: the indexer
 * cache must hold exactly the sequence's tokens before the step; more is the
 * leftover of a rejected verify and is rewound, fewer means rows were never
 * written and is an error), when idx_written is given ([rows / rows_per_seq]
 * int32, one count per sequence of rows_per_seq consecutive rows, which must
 * have the consecutive positions p0, p0+1, ...): a sequence whose count is
 * below p0 is not written and is recorded as DSA_DEVERR_BEHIND; otherwise
 * its rows are written and its count becomes p0 + rows_per_seq (a count
 * above p0 is rewound).  rows_per_seq in [1, 32] and dividing rows when
 * idx_written is given (ignored otherwise).
 */
dsa_status dsa_indexer_write(const dsa_rows *rows, const uint16_t *k_raw, const uint16_t *ln_w,
                             const uint16_t *ln_b, float eps, const uint16_t *gate,
                             const int64_t *idx_base, uint16_t *idx_k, uint16_t *idx_gate,
                             int64_t idx_tokens, int32_t index_dim, int32_t *idx_written,
                             int32_t rows_per_seq, void *stream);

/*
 * Batched projection for the K-token verify: the K rows of one sequence sweep
 * a BF16 weight once ("glm5next_dsa/layer.rs": the gemm helper,
 * C[M, N] = A[M, K] @ B[N, K]^T, and the decode_k notes on
 * dense_gemv_bf16_batchm -- one weight read for 2..16 rows, each row
 * bit-identical to a single-row call).
 *   c[m][n] = sum_k a[m][k] * b[n][k]          m < m_rows, n < n_out
 *   a [m_rows][k] bf16, row-major (k contiguous), 16-byte aligned
 *   b [n_out][k]  bf16 weight, row-major, 16-byte aligned
 *   c [m_rows][n_out] bf16 (c_fp32 = 0, round to nearest even) or fp32
 *     (c_fp32 = 1), 4-byte aligned
 * m_rows in [1, 16] (DSA_ERR_UNSUPPORTED above); k >= 8 and a multiple of 8
 * (16-byte row strides); n_out >= 1; DSA_ERR_INVALID_ARG otherwise.
 * Numerics: the bf16 products are exact and accumulate in FP32 on the tensor
 * cores in 64-element blocks of k, in order; when the weight has few rows the
 * k range is split (the split depends only on n_out, k and the device's SM
 * count) and the FP32 partial sums are added in order.  A row's result is a
 * function of that row of a and of b only: bit-identical whatever m_rows is
 * and whatever the other rows hold.  The split partials pass through the
 * caller's workspace of dsa_dense_mm_workspace_bytes(n_out, k) bytes (0: none
 * needed), 256-byte aligned (DSA_ERR_WORKSPACE otherwise).
 */
dsa_status dsa_dense_mm_bf16(const uint16_t *a, const uint16_t *b, void *c, int32_t m_rows,
                             int32_t n_out, int32_t k, int32_t c_fp32, void *workspace,
                             size_t workspace_bytes, void *stream);

/* The number of k ranges dsa_dense_mm_bf16 splits an n_out x k weight into on
 * a device with num_sms SMs (host arithmetic only; 0 on bad arguments).  One
 * range when the 128-row weight tiles alone reach num_sms, else enough ranges
 * to, each at least four 64-element blocks of k long. */
int32_t dsa_dense_mm_splits(int32_t n_out, int32_t k, int32_t num_sms);

/* Workspace bytes dsa_dense_mm_bf16 needs on the current device for a weight
 * of n_out x k (0 when it needs none or on bad arguments). */
size_t dsa_dense_mm_workspace_bytes(int32_t n_out, int32_t k);

/*
 * Read the sticky device error word of the current device: *code_out is the
 * first DSA_DEVERR_* recorded since the last reset (0 if none), *row_out the
 * row it concerned and *count_out how many errors were recorded.  Any out
 * pointer may be NULL.  This call synchronises the device.  reset != 0 clears
 * the word.  Returns DSA_ERR_DEVICE when an error was recorded, else DSA_OK
 * (or DSA_ERR_CUDA).
 */
dsa_status dsa_get_error(int32_t *code_out, int32_t *row_out, int32_t *count_out, int32_t reset);

/* Block-table entries the paged gather can index for k rows starting at
 * seq_len, plus one of slack: (seq_len + k) / block_size + 2, a block size of
 * 0 counted as 1 ("glm5next_dsa/layer.rs", bt_entries_needed). */
int64_t dsa_bt_entries_needed(int64_t seq_len, int64_t k, int64_t block_size);

/*
 * Limit, in nanoseconds of wall time, on every pipeline wait inside the
 * kernels launched after this call (0 restores the default, 500 ms).  A wait
 * that runs out records DSA_DEVERR_TIMEOUT, the CTA stops its pipeline and
 * its results are zero; the CTA still waits for its own copies and MMAs in
 * flight (that drain keeps its own 500 ms limit) before it exits, so a short
 * limit never leaves work running behind the call.  Meant for tests of the
 * timeout path and for callers that prefer an early error to a long stall;
 * process-wide.  No counterpart on the pages.
 */
dsa_status dsa_set_wait_limit_ns(uint64_t limit_ns);
uint64_t dsa_get_wait_limit_ns(void);

/* Static text for a status code. */
const char *dsa_status_string(dsa_status status);

/* DSA_ABI_VERSION of the loaded library. */
int32_t dsa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
