// dsa_internal.h -- host-side launch interfaces between the C ABI layer
// (dsa_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// Launch attribute that lets a kernel start before its stream predecessor
// finishes (it then waits with griddepcontrol.wait where it needs to).
inline cudaLaunchAttribute dependent_launch_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Device address of the sticky error word on the current device (nullptr on
// failure); kernels receive it as an argument.
int* device_error_word();

// Bound on every pipeline wait in the kernels (wall time); dsa_set_wait_limit_ns
// changes it for later launches.
constexpr uint64_t kDefaultWaitNs = 500ull * 1000ull * 1000ull;
uint64_t wait_limit_ns();
// Bound on the drain at the end of a CTA -- the waits for its own TMA copies
// and MMAs still in flight before TMEM is released and the CTA exits.  It is
// never shortened: a pipeline wait that gave up must not leave a copy or an
// MMA running behind the CTA.
constexpr uint64_t kDrainWaitNs = 500ull * 1000ull * 1000ull;

struct LatentWriteParams {
  dsa_rows rows;
  const uint16_t* kv_a;
  const uint16_t* norm_w;
  uint8_t* pool;
  int64_t nslots;
  float eps;
  float inv_scale;  // fl32(1 / kv_scale)
  int* err;
};
cudaError_t launch_latent_write(const LatentWriteParams& p, cudaStream_t stream);

struct IndexParams {
  const int32_t* seq_lens;
  const float* q_idx;
  const float* head_w;
  const uint16_t* gate;
  const int64_t* idx_base;
  const int32_t* idx_written;  // [sequences] rows written per sequence, or nullptr
  float* scores;
  int* err;
  int64_t idx_tokens;
  int32_t rows;
  int32_t rows_per_seq;   // caller's sequence group size G
  int32_t sub_rows;       // rows per launch group (<= G, npad <= 256)
  int32_t subs_per_seq;   // ceil(G / sub_rows)
  int32_t heads;
  int32_t dim;            // 64 or 128
  int32_t npad;           // sub_rows*heads rounded up to a multiple of 16
  int32_t max_len;
  int32_t ctas;           // persistent CTAs (one wave)
  int32_t direct;         // 1: direct_tiles tiles per CTA, grid (tile block, group)
  int32_t direct_tiles;
  int32_t stages;         // smem pipeline depth
  uint32_t tmem_cols;
  uint32_t smem_bytes;
  uint64_t wait_ns;
  int32_t inputs_early;   // inputs complete before the kernel before started: only the
                          // score stores (and the exit) wait for it
};
// Fills in direct / ctas / stages / tmem_cols / smem_bytes from the shape.
void plan_index_scores(IndexParams& p, int num_sms);
cudaError_t launch_index_scores(const IndexParams& p, const CUtensorMap& kmap,
                                cudaStream_t stream);

struct TopkParams {
  const int32_t* seq_lens;
  const float* scores;
  int32_t* sel;
  int* err;
  int32_t rows;
  int32_t max_len;
  int32_t topk;
  int32_t cluster;   // CTAs per row (one thread-block cluster)
};
// CTAs per row (one cluster) for `rows` rows of max_len keys.
int topk_cluster_size(int32_t max_len, int32_t rows, int num_sms);
size_t topk_smem_bytes(int32_t max_len, int cluster);
cudaError_t launch_select_topk(const TopkParams& p, cudaStream_t stream);

struct PoolSelectParams {
  const uint32_t* positions;  // [rows] q_pos
  const float* scores;        // [rows][max_pools]
  const uint8_t* valid;       // row r at valid + r*valid_stride, [max_pools]
  int32_t* sel_pools;         // [rows][select_k]
  int32_t* sel_tokens;        // [rows][out_width]
  int32_t rows;
  int32_t max_pools;
  int32_t valid_stride;
  int32_t kp;
  int32_t select_k;
  int32_t out_width;
};
size_t select_pools_smem_bytes(int32_t max_pools);
cudaError_t launch_select_pools(const PoolSelectParams& p, cudaStream_t stream);
cudaError_t launch_expand_selection(const PoolSelectParams& p, cudaStream_t stream);

struct IndexerWriteParams {
  const uint32_t* positions;
  const int32_t* seq_lens;
  const int64_t* idx_base;
  const uint16_t* k_raw;   // [rows][dim] bf16
  const uint16_t* ln_w;    // [dim] bf16
  const uint16_t* ln_b;    // [dim] bf16
  const uint16_t* gate;    // [rows] bf16 or nullptr
  uint16_t* idx_k;         // [idx_tokens][dim] bf16
  uint16_t* idx_gate;      // [idx_tokens] bf16
  int32_t* idx_written;    // [sequences] rows written per sequence, or nullptr
  int64_t idx_tokens;
  int32_t rows;
  int32_t rows_per_seq;    // rows of one sequence (consecutive positions), with idx_written
  int32_t dim;
  float eps;
  int* err;
};
cudaError_t launch_indexer_write(const IndexerWriteParams& p, cudaStream_t stream);

struct DenseMmParams {
  const uint16_t* a;      // [m][k] bf16 activations
  const uint16_t* b;      // [n][k] bf16 weight
  void* c;                // [m][n] bf16 or fp32
  float* part;            // workspace: [splits][m][n] fp32 partials (splits > 1)
  int* err;
  int32_t m, n, k;
  int32_t c_fp32;
  int32_t tiles;          // 128-row weight tiles
  int32_t kblocks;        // 64-element K blocks
  int32_t kb_per_split;   // K blocks per CTA
  int32_t splits;         // K ranges per weight tile
  uint64_t wait_ns;
};
// Fills in tiles / kblocks / kb_per_split / splits from (n, k) and the SM count.
void plan_dense_mm(DenseMmParams& p, int num_sms);
size_t dense_mm_workspace_bytes(int32_t n, int32_t k, int num_sms);
cudaError_t launch_dense_mm(const DenseMmParams& p, const CUtensorMap& wmap,
                            const CUtensorMap& amap, cudaStream_t stream);

struct DecodeParams {
  dsa_rows rows;
  const uint16_t* q;
  const uint8_t* pool;
  int64_t nslots;
  const int32_t* sel;
  uint16_t* out;
  float* lse;
  uint16_t* part_o; // workspace: [rows][head groups][splits][64][512] fp16 O / l of the split
  float* part_ml;   // workspace: [rows][head groups][splits][64] (max, sum)
  int* err;
  int32_t topk;
  int32_t heads;
  int32_t splits;
  int32_t split_len;   // selection entries per split (cluster form)
  uint64_t wait_ns;    // pipeline wait limit
  float kv_scale;
  float sm_scale;
  int32_t q_early;     // CTAs (in launch order) that load q before the dependency wait
  int32_t long_splits; // caller's choice: 512-entry splits at up to 64 heads (set before planning)
  int32_t num_sms;     // SMs of the device (the merge kernel's launch shape only)
};
// Split count / length of the gather-attend (a function of topk, heads and
// long_splits only).
void plan_mla_decode_tc(DecodeParams& p);
size_t mla_decode_tc_workspace_bytes(int32_t rows, int32_t heads, int32_t topk);
void mla_decode_tc_bind_workspace(DecodeParams& p, void* workspace);
// Split kernel (tcgen05) followed by the merge kernel.  `pmap` describes the
// latent pool [nslots][512] bytes for 128-byte x 1-row TMA gathers.
cudaError_t launch_mla_decode_tc(const DecodeParams& p, const CUtensorMap& pmap,
                                 cudaStream_t stream);

}  // namespace dsa
