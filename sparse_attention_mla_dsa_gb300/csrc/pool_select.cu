// pool_select.cu -- the pool-compressed selector's specified half: the top
// pools of each row over caller-supplied pool scores, and their expansion to
// token indices with the visible tail.
//
// "glm5next_dsa/layer.rs", the notes above batch_select_enabled and on
// select_rows_batched: pool p (tokens [p*KP, (p+1)*KP)) is a candidate for
// row r only when it is complete (pool_valid[p]) and its last token is visible
// to the row ((p+1)*KP - 1 <= q_pos[r]); the pools are taken under the total
// order (score DESC, then pool index ASC); the per-row count
// row_select_k = min(select_k, (q_pos[r] + 1) / KP) sets both how many pools
// are taken and where the visible tail starts (row_select_k * KP).
//
// select_pools_kernel: one CTA per row.  Only the row's own pools p <
// (q_pos+1)/KP can be candidates, so only they are read.  Each becomes a
// 64-bit key, the score's order-preserving key in the high half and the
// inverted pool index in the low half (0 for a non-candidate), and a
// descending bitonic sort in shared memory puts the candidates in the total
// order; the first row_select_k of them are the row's pools.
// expand_selection_kernel: one thread per output entry.
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kSortThreads = 512;
constexpr int kExpandThreads = 256;

__device__ __forceinline__ int64_t row_select_k(int64_t q_pos, int32_t kp, int32_t select_k) {
  const int64_t visible = q_pos + 1 >= 0 ? (q_pos + 1) / kp : 0;
  return visible < select_k ? visible : select_k;
}

__global__ void __launch_bounds__(kSortThreads) select_pools_kernel(const PoolSelectParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint64_t* key = reinterpret_cast<uint64_t*>(smem_raw);
  const int r = blockIdx.x, tid = threadIdx.x;
  grid_dep_wait();  // scores, validity and positions may come from the kernel before
  grid_dep_launch();
  const int64_t q_pos = static_cast<int64_t>(p.positions[r]);
  const int64_t k = row_select_k(q_pos, p.kp, p.select_k);
  const int64_t visible = (q_pos + 1) / p.kp;
  const int own = static_cast<int>(visible < p.max_pools ? visible : p.max_pools);
  int n = 1;
  while (n < own) n <<= 1;
  const float* sc = p.scores + static_cast<int64_t>(r) * p.max_pools;
  const uint8_t* vd = p.valid + static_cast<int64_t>(r) * p.valid_stride;
  for (int i = tid; i < n; i += kSortThreads) {
    uint64_t v = 0;
    if (i < own && vd[i] != 0)
      v = (static_cast<uint64_t>(order_key(sc[i])) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(i));
    key[i] = v;
  }
  __syncthreads();
  // Descending bitonic sort of n keys.
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n; i += kSortThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const uint64_t a = key[i], b = key[j];
          const bool desc = (i & size) == 0;
          if (desc ? a < b : a > b) {
            key[i] = b;
            key[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  int32_t* out = p.sel_pools + static_cast<int64_t>(r) * p.select_k;
  for (int i = tid; i < p.select_k; i += kSortThreads) {
    int32_t v = -1;
    if (i < k && i < n && key[i] != 0)
      v = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key[i] & 0xFFFFFFFFu));
    out[i] = v;
  }
}

__global__ void __launch_bounds__(kExpandThreads) expand_selection_kernel(const PoolSelectParams p) {
  const int r = blockIdx.y;
  const int i = blockIdx.x * kExpandThreads + threadIdx.x;
  grid_dep_wait();  // the pools come from the kernel before
  grid_dep_launch();
  if (i >= p.out_width) return;
  const int64_t q_pos = static_cast<int64_t>(p.positions[r]);
  const int64_t k = row_select_k(q_pos, p.kp, p.select_k);
  const int64_t slot = i / p.kp;
  int64_t tok = -1;
  if (slot < k) {
    const int32_t pool = p.sel_pools[static_cast<int64_t>(r) * p.select_k + slot];
    if (pool >= 0) tok = static_cast<int64_t>(pool) * p.kp + i % p.kp;
  } else {
    // the visible tail: tokens after the last complete pool, up to q_pos
    const int64_t tail_start = ((q_pos + 1) / p.kp) * p.kp;
    const int64_t t = tail_start + (i - k * p.kp);
    if (t <= q_pos) tok = t;
  }
  p.sel_tokens[static_cast<int64_t>(r) * p.out_width + i] = static_cast<int32_t>(tok);
}

}  // namespace

size_t select_pools_smem_bytes(int32_t max_pools) {
  size_t n = 1;
  while (n < static_cast<size_t>(max_pools)) n <<= 1;
  return n * sizeof(uint64_t);
}

cudaError_t launch_select_pools(const PoolSelectParams& p, cudaStream_t stream) {
  const size_t smem = select_pools_smem_bytes(p.max_pools);
  cudaError_t e = cudaFuncSetAttribute(select_pools_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows, 1, 1);
  cfg.blockDim = dim3(kSortThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_pools_kernel, p);
}

cudaError_t launch_expand_selection(const PoolSelectParams& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.out_width + kExpandThreads - 1) / kExpandThreads, p.rows, 1);
  cfg.blockDim = dim3(kExpandThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, expand_selection_kernel, p);
}

}  // namespace dsa
