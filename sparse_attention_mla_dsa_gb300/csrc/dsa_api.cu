// dsa_api.cu -- the C ABI declared in include/dsa.h: argument validation,
// launch planning, the device error word and the TMA descriptor of the key
// arena.  No call here allocates, frees, copies host<->device or synchronises
// (except dsa_get_error, which says so).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

// The sticky device error word (one per device that loads the library).
__device__ int g_error_word[4];

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int* err = nullptr;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    d.err = static_cast<int*>(p);
    d.ready = true;
  }
  return &d;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode_tiled == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode_tiled;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

dsa_status check_rows(const dsa_rows* rows, bool need_table) {
  if (rows == nullptr || rows->rows < 1 || rows->seq_lens == nullptr) return DSA_ERR_INVALID_ARG;
  if (rows->rows > 65535) return DSA_ERR_UNSUPPORTED;
  if (need_table) {
    if (rows->block_table == nullptr || rows->block_size < 1 || rows->max_blocks_per_seq < 1 ||
        rows->bt_stride < 0)
      return DSA_ERR_INVALID_ARG;
    if (rows->bt_stride != 0 && rows->bt_stride < rows->max_blocks_per_seq)
      return DSA_ERR_INVALID_ARG;
  }
  return DSA_OK;
}

dsa_status launched(cudaError_t e) { return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA; }

}  // namespace

int* device_error_word() {
  const DeviceInfo* d = device_info();
  return d ? d->err : nullptr;
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

}  // namespace dsa

using namespace dsa;

extern "C" {

dsa_status dsa_latent_write(const dsa_rows* rows, const uint16_t* kv_a, const uint16_t* norm_w,
                            uint8_t* pool, int64_t nslots, int32_t latent_dim, float eps,
                            float kv_scale, void* stream) {
  dsa_status st = check_rows(rows, rows != nullptr && rows->positions != nullptr);
  if (st != DSA_OK) return st;
  if (rows->slots == nullptr || kv_a == nullptr || norm_w == nullptr || pool == nullptr ||
      nslots < 1)
    return DSA_ERR_INVALID_ARG;
  if (latent_dim != DSA_LATENT_DIM) return DSA_ERR_UNSUPPORTED;
  if (!(kv_scale > 0.0f) || !(eps >= 0.0f)) return DSA_ERR_INVALID_ARG;
  if (!aligned(kv_a, 8) || !aligned(norm_w, 8) || !aligned(pool, 4)) return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  LatentWriteParams p{};
  p.rows = *rows;
  p.kv_a = kv_a;
  p.norm_w = norm_w;
  p.pool = pool;
  p.nslots = nslots;
  p.eps = eps;
  p.inv_scale = 1.0f / kv_scale;
  p.err = dev->err;
  return launched(launch_latent_write(p, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_index_scores(const dsa_rows* rows, const float* q_idx, const float* head_w,
                            const uint16_t* idx_k, const uint16_t* idx_gate, int64_t idx_tokens,
                            const int64_t* idx_base, int32_t index_heads, int32_t index_dim,
                            int32_t rows_per_seq, int32_t max_len, float* scores,
                            const int32_t* idx_written, void* stream) {
  return dsa_index_scores_ex(rows, q_idx, head_w, idx_k, idx_gate, idx_tokens, idx_base,
                             index_heads, index_dim, rows_per_seq, max_len, scores, idx_written,
                             0u, stream);
}

dsa_status dsa_index_scores_ex(const dsa_rows* rows, const float* q_idx, const float* head_w,
                               const uint16_t* idx_k, const uint16_t* idx_gate, int64_t idx_tokens,
                               const int64_t* idx_base, int32_t index_heads, int32_t index_dim,
                               int32_t rows_per_seq, int32_t max_len, float* scores,
                               const int32_t* idx_written, uint32_t flags, void* stream) {
  if ((flags & ~DSA_INDEX_INPUTS_BEFORE_PREDECESSOR) != 0) return DSA_ERR_INVALID_ARG;
  dsa_status st = check_rows(rows, false);
  if (st != DSA_OK) return st;
  if (q_idx == nullptr || head_w == nullptr || idx_k == nullptr || idx_gate == nullptr ||
      idx_base == nullptr || scores == nullptr || idx_tokens < 1 || max_len < 0)
    return DSA_ERR_INVALID_ARG;
  if (rows_per_seq < 1 || rows->rows % rows_per_seq != 0) return DSA_ERR_INVALID_ARG;
  if (index_dim != 64 && index_dim != 128) return DSA_ERR_UNSUPPORTED;
  if (index_heads < 1 || index_heads > 256) return DSA_ERR_UNSUPPORTED;
  if (idx_tokens > 0x7FFFFFFFLL) return DSA_ERR_UNSUPPORTED;
  if (!aligned(idx_k, 16) || !aligned(q_idx, 16)) return DSA_ERR_INVALID_ARG;
  if (max_len == 0) return DSA_OK;
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  auto encode = encode_tiled();
  if (encode == nullptr) return DSA_ERR_CUDA;

  IndexParams p{};
  p.seq_lens = rows->seq_lens;
  p.q_idx = q_idx;
  p.head_w = head_w;
  p.gate = idx_gate;
  p.idx_base = idx_base;
  p.idx_written = idx_written;
  p.scores = scores;
  p.err = dev->err;
  p.idx_tokens = idx_tokens;
  p.rows = rows->rows;
  p.rows_per_seq = rows_per_seq;
  // Rows of one sequence share each key tile in groups of at most 64 score
  // columns (a wider group makes the per-token epilogue, not HBM, the limit,
  // and its q operand leaves room for one CTA per SM; the groups of a
  // sequence run side by side and share the key tiles through L2); a head
  // count that is not a multiple of 16 runs one row per launch group so that
  // no 16-column TMEM load straddles two rows.
  int sub = 64 / index_heads;
  if (index_heads % 16 != 0) sub = 1;
  sub = sub < 1 ? 1 : (sub > 32 ? 32 : sub);
  if (sub > rows_per_seq) sub = rows_per_seq;
  p.sub_rows = sub;
  p.subs_per_seq = (rows_per_seq + sub - 1) / sub;
  p.heads = index_heads;
  p.dim = index_dim;
  p.npad = ((sub * index_heads + 15) / 16) * 16;
  p.max_len = max_len;
  p.wait_ns = wait_limit_ns();
  p.inputs_early = (flags & DSA_INDEX_INPUTS_BEFORE_PREDECESSOR) != 0 ? 1 : 0;
  plan_index_scores(p, dev->num_sms);

  // Key arena [idx_tokens, index_dim] bf16, boxes of 128 tokens x 64 dims
  // (128 bytes, the swizzle span); rows past the arena read as zero.
  CUtensorMap kmap;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(index_dim), static_cast<cuuint64_t>(idx_tokens)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(index_dim) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estride[2] = {1, 1};
  CUresult cr = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(idx_k),
                       gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return DSA_ERR_INVALID_ARG;
  return launched(launch_index_scores(p, kmap, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_select_topk(const dsa_rows* rows, const float* scores, int32_t max_len,
                           int32_t topk, int32_t* sel, void* stream) {
  dsa_status st = check_rows(rows, false);
  if (st != DSA_OK) return st;
  if (scores == nullptr || sel == nullptr || max_len < 0) return DSA_ERR_INVALID_ARG;
  if (topk < 1 || topk > 65536) return DSA_ERR_UNSUPPORTED;
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  TopkParams p{};
  p.seq_lens = rows->seq_lens;
  p.scores = scores;
  p.sel = sel;
  p.err = dev->err;
  p.rows = rows->rows;
  p.max_len = max_len;
  p.topk = topk;
  p.cluster = topk_cluster_size(max_len, rows->rows, dev->num_sms);
  if (topk_smem_bytes(max_len, p.cluster) > 227u * 1024u) return DSA_ERR_UNSUPPORTED;
  return launched(launch_select_topk(p, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_mla_decode_fp8(const dsa_rows* rows, const uint16_t* q, const uint8_t* pool,
                              int64_t nslots, const int32_t* sel, int32_t topk, int32_t heads,
                              int32_t latent_dim, float kv_scale, float sm_scale, uint16_t* out,
                              float* lse_or_null, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return dsa_mla_decode_fp8_ex(rows, q, pool, nslots, sel, topk, heads, latent_dim, kv_scale,
                               sm_scale, out, lse_or_null, workspace, workspace_bytes, 0u, stream);
}

dsa_status dsa_mla_decode_fp8_ex(const dsa_rows* rows, const uint16_t* q, const uint8_t* pool,
                                 int64_t nslots, const int32_t* sel, int32_t topk, int32_t heads,
                                 int32_t latent_dim, float kv_scale, float sm_scale,
                                 uint16_t* out, float* lse_or_null, void* workspace,
                                 size_t workspace_bytes, uint32_t flags, void* stream) {
  if ((flags & ~static_cast<uint32_t>(DSA_DECODE_Q_BEFORE_PREDECESSOR | DSA_DECODE_LONG_SPLITS)) != 0u)
    return DSA_ERR_INVALID_ARG;
  dsa_status st = check_rows(rows, true);
  if (st != DSA_OK) return st;
  if (q == nullptr || pool == nullptr || sel == nullptr || out == nullptr || nslots < 1)
    return DSA_ERR_INVALID_ARG;
  if (latent_dim != DSA_LATENT_DIM || nslots > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (heads < 16 || heads % 16 != 0 || heads > 4096) return DSA_ERR_UNSUPPORTED;
  if (topk < 1 || topk > 65536) return DSA_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(pool, 16) || !aligned(out, 8)) return DSA_ERR_INVALID_ARG;
  {
    // out: device memory, or page-locked host memory the device reaches at
    // the same address; anything else is refused before a kernel could touch it.
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, out) != cudaSuccess) {
      cudaGetLastError();  // not sticky: clear it for the caller
      return DSA_ERR_INVALID_ARG;
    }
    const bool on_device = a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
    const bool mapped_host = a.type == cudaMemoryTypeHost && a.devicePointer == out;
    if (!on_device && !mapped_host) return DSA_ERR_INVALID_ARG;
  }
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  DecodeParams p{};
  p.rows = *rows;
  p.q = q;
  p.pool = pool;
  p.nslots = nslots;
  p.sel = sel;
  p.out = out;
  p.lse = lse_or_null;
  p.topk = topk;
  p.heads = heads;
  p.err = dev->err;
  p.kv_scale = kv_scale;
  p.sm_scale = sm_scale;
  p.wait_ns = wait_limit_ns();
  // Only CTAs of the first wave can be waiting on the kernel before: later
  // ones start after it has finished, and for them the default order (q and
  // the selection loaded together after the wait) is the faster one.
  p.q_early = (flags & DSA_DECODE_Q_BEFORE_PREDECESSOR) != 0u ? dev->num_sms : 0;
  p.long_splits = (flags & DSA_DECODE_LONG_SPLITS) != 0u ? 1 : 0;
  p.num_sms = dev->num_sms;
  plan_mla_decode_tc(p);
  const size_t need = mla_decode_tc_workspace_bytes(rows->rows, heads, topk);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return DSA_ERR_WORKSPACE;
  mla_decode_tc_bind_workspace(p, workspace);
  auto encode = encode_tiled();
  if (encode == nullptr) return DSA_ERR_CUDA;
  // Latent pool [nslots][512] bytes; the gather reads 128-byte x 1-row boxes
  // (tile::gather4: four rows per copy) with the 128-byte swizzle; rows
  // outside the pool read as zero.
  CUtensorMap pmap;
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(DSA_LATENT_DIM), static_cast<cuuint64_t>(nslots)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(DSA_LATENT_DIM)};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estride[2] = {1, 1};
  CUresult cr = encode(&pmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(pool), gdim,
                       gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return DSA_ERR_INVALID_ARG;
  return launched(launch_mla_decode_tc(p, pmap, static_cast<cudaStream_t>(stream)));
}

size_t dsa_workspace_bytes(int32_t rows, int32_t heads, int32_t topk) {
  if (rows < 1 || heads < 1 || topk < 1) return 0;
  return mla_decode_tc_workspace_bytes(rows, heads, topk);
}

dsa_status dsa_select_pools(const dsa_rows* rows, const float* pool_scores, int32_t max_pools,
                            const uint8_t* pool_valid, int32_t valid_stride, int32_t kp,
                            int32_t select_k, int32_t* sel_pools, void* stream) {
  dsa_status st = check_rows(rows, false);
  if (st != DSA_OK) return st;
  if (rows->positions == nullptr || pool_scores == nullptr || pool_valid == nullptr ||
      sel_pools == nullptr || kp < 1 || select_k < 1 || max_pools < 1 || valid_stride < 0 ||
      (valid_stride != 0 && valid_stride < max_pools))
    return DSA_ERR_INVALID_ARG;
  if (max_pools > DSA_MAX_POOLS) return DSA_ERR_UNSUPPORTED;
  PoolSelectParams p{};
  p.positions = rows->positions;
  p.scores = pool_scores;
  p.valid = pool_valid;
  p.sel_pools = sel_pools;
  p.rows = rows->rows;
  p.max_pools = max_pools;
  p.valid_stride = valid_stride;
  p.kp = kp;
  p.select_k = select_k;
  return launched(launch_select_pools(p, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_expand_selection(const dsa_rows* rows, const int32_t* sel_pools, int32_t kp,
                                int32_t select_k, int32_t* sel_tokens, int32_t out_width,
                                void* stream) {
  dsa_status st = check_rows(rows, false);
  if (st != DSA_OK) return st;
  if (rows->positions == nullptr || sel_pools == nullptr || sel_tokens == nullptr || kp < 1 ||
      select_k < 1)
    return DSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(out_width) < static_cast<int64_t>(select_k) * kp + kp - 1)
    return DSA_ERR_INVALID_ARG;
  PoolSelectParams p{};
  p.positions = rows->positions;
  p.sel_pools = const_cast<int32_t*>(sel_pools);
  p.sel_tokens = sel_tokens;
  p.rows = rows->rows;
  p.kp = kp;
  p.select_k = select_k;
  p.out_width = out_width;
  return launched(launch_expand_selection(p, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_indexer_write(const dsa_rows* rows, const uint16_t* k_raw, const uint16_t* ln_w,
                             const uint16_t* ln_b, float eps, const uint16_t* gate,
                             const int64_t* idx_base, uint16_t* idx_k, uint16_t* idx_gate,
                             int64_t idx_tokens, int32_t index_dim, int32_t* idx_written,
                             int32_t rows_per_seq, void* stream) {
  dsa_status st = check_rows(rows, false);
  if (st != DSA_OK) return st;
  if (rows->positions == nullptr || k_raw == nullptr || ln_w == nullptr || ln_b == nullptr ||
      idx_base == nullptr || idx_k == nullptr || idx_tokens < 1)
    return DSA_ERR_INVALID_ARG;
  if (gate != nullptr && idx_gate == nullptr) return DSA_ERR_INVALID_ARG;
  if (index_dim != 64 && index_dim != 128) return DSA_ERR_UNSUPPORTED;
  if (!(eps >= 0.0f)) return DSA_ERR_INVALID_ARG;
  if (!aligned(k_raw, 8) || !aligned(idx_k, 8)) return DSA_ERR_INVALID_ARG;
  if (idx_written != nullptr &&
      (rows_per_seq < 1 || rows_per_seq > 32 || rows->rows % rows_per_seq != 0))
    return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  IndexerWriteParams p{};
  p.idx_written = idx_written;
  p.rows_per_seq = idx_written != nullptr ? rows_per_seq : 1;
  p.positions = rows->positions;
  p.seq_lens = rows->seq_lens;
  p.idx_base = idx_base;
  p.k_raw = k_raw;
  p.ln_w = ln_w;
  p.ln_b = ln_b;
  p.gate = gate;
  p.idx_k = idx_k;
  p.idx_gate = idx_gate;
  p.idx_tokens = idx_tokens;
  p.rows = rows->rows;
  p.dim = index_dim;
  p.eps = eps;
  p.err = dev->err;
  return launched(launch_indexer_write(p, static_cast<cudaStream_t>(stream)));
}

int32_t dsa_dense_mm_splits(int32_t n_out, int32_t k, int32_t num_sms) {
  if (n_out < 1 || k < 8 || k % 8 != 0 || num_sms < 1) return 0;
  DenseMmParams p{};
  p.n = n_out;
  p.k = k;
  plan_dense_mm(p, num_sms);
  return p.splits;
}

size_t dsa_dense_mm_workspace_bytes(int32_t n_out, int32_t k) {
  if (n_out < 1 || k < 8 || k % 8 != 0) return 0;
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return 0;
  return dense_mm_workspace_bytes(n_out, k, dev->num_sms);
}

dsa_status dsa_dense_mm_bf16(const uint16_t* a, const uint16_t* b, void* c, int32_t m_rows,
                             int32_t n_out, int32_t k, int32_t c_fp32, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (a == nullptr || b == nullptr || c == nullptr) return DSA_ERR_INVALID_ARG;
  if (m_rows < 1 || n_out < 1 || k < 8 || k % 8 != 0) return DSA_ERR_INVALID_ARG;
  if (m_rows > 16) return DSA_ERR_UNSUPPORTED;
  if (c_fp32 != 0 && c_fp32 != 1) return DSA_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 4)) return DSA_ERR_INVALID_ARG;
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  auto encode = encode_tiled();
  if (encode == nullptr) return DSA_ERR_CUDA;

  DenseMmParams p{};
  p.a = a;
  p.b = b;
  p.c = c;
  p.err = dev->err;
  p.m = m_rows;
  p.n = n_out;
  p.k = k;
  p.c_fp32 = c_fp32;
  p.wait_ns = wait_limit_ns();
  plan_dense_mm(p, dev->num_sms);
  if (p.splits > 1) {
    const size_t need = static_cast<size_t>(p.splits) * m_rows * static_cast<size_t>(n_out) * 4;
    if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
      return DSA_ERR_WORKSPACE;
    p.part = static_cast<float*>(workspace);
  }

  // Weight [n_out][k] and activations [m_rows][k], bf16, boxes of 64 of k
  // (128 bytes, the swizzle span) by 128 weight rows / 16 activation rows;
  // rows and columns past the tensors read as zero.
  CUtensorMap wmap, amap;
  cuuint64_t wdim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(n_out)};
  cuuint64_t adim[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(m_rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(k) * 2};
  cuuint32_t wbox[2] = {64, 128};
  cuuint32_t abox[2] = {64, 16};
  cuuint32_t estride[2] = {1, 1};
  CUresult cr = encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(b), wdim,
                       gstride, wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return DSA_ERR_INVALID_ARG;
  cr = encode(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a), adim, gstride,
              abox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return DSA_ERR_INVALID_ARG;
  return launched(launch_dense_mm(p, wmap, amap, static_cast<cudaStream_t>(stream)));
}

dsa_status dsa_get_error(int32_t* code_out, int32_t* row_out, int32_t* count_out, int32_t reset) {
  const DeviceInfo* dev = device_info();
  if (dev == nullptr) return DSA_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
  int word[4] = {0, 0, 0, 0};
  if (cudaMemcpy(word, dev->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (reset) {
    if (cudaMemset(dev->err, 0, sizeof word) != cudaSuccess) return DSA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return DSA_ERR_CUDA;
  }
  if (code_out) *code_out = word[0];
  if (row_out) *row_out = word[1];
  if (count_out) *count_out = word[2];
  return word[0] != 0 ? DSA_ERR_DEVICE : DSA_OK;
}

int64_t dsa_bt_entries_needed(int64_t seq_len, int64_t k, int64_t block_size) {
  const int64_t bs = block_size > 0 ? block_size : 1;
  return (seq_len + k) / bs + 2;
}

const char* dsa_status_string(dsa_status status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or size";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_DEVICE: return "device-side error recorded";
    case DSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

dsa_status dsa_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns != 0 ? limit_ns : kDefaultWaitNs, std::memory_order_relaxed);
  return DSA_OK;
}

uint64_t dsa_get_wait_limit_ns(void) { return wait_limit_ns(); }

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

}  // extern "C"
