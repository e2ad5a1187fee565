// select_topk.cu -- S2: per-row top-k of the indexer scores.
//
// "glm5next_dsa/layer.rs", notes on batch_select_enabled / select_rows_batched:
// the selection is taken under a total order (score DESC, then index ASC), so
// the top-k set is unique; each row's result is a function of its own scores.
//
// One CTA of 1024 threads per row: a three-digit radix select (11 + 11 + 10
// bits) over an order-preserving 32-bit key finds the k-th largest key T and
// how many keys equal to T belong to the selection; a final in-order pass then
// writes every token with key > T plus the lowest-index tokens with key == T,
// in ascending token order (block-wide prefix sums keep the order).
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 8;  // consecutive tokens per thread in the output pass

// Larger float -> larger unsigned key; -0.0 is folded onto +0.0 first.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix sum over the CTA; also returns the total.  Contains
// __syncthreads, so every thread must call it.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    warp_tot[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp ? warp_tot[warp - 1] : 0;
  total = warp_tot[kWarps - 1];
  __syncthreads();  // warp_tot may be reused right after
  return before + x - v;
}

__global__ void __launch_bounds__(kThreads) select_topk_kernel(TopkParams p) {
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  __shared__ int hist[2048];
  __shared__ int warp_tot[kWarps];
  __shared__ int found_bin, found_above;

  int len = p.seq_lens[r];
  if (len < 0 || len > p.max_len) {
    if (tid == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }
  const float* row = p.scores + static_cast<int64_t>(r) * p.max_len;
  int32_t* out = p.sel + static_cast<int64_t>(r) * p.topk;
  const int want = min(p.topk, len);

  if (len <= p.topk) {  // everything visible is selected
    for (int i = tid; i < p.topk; i += kThreads) out[i] = i < len ? i : -1;
    return;
  }

  // ---- radix select: find the key T of the want-th largest and how many
  // keys equal to T are taken (`remaining` after the last digit).
  uint32_t prefix = 0, prefix_mask = 0;
  int remaining = want;
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int b = tid; b < nb; b += kThreads) hist[b] = 0;
    __syncthreads();
    for (int t = tid; t < len; t += kThreads) {
      const uint32_t key = order_key(row[t]);
      if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1);
    }
    __syncthreads();
    // Thread i owns bins nb-1-2i and nb-2-2i (descending), so an exclusive
    // scan gives the count of keys in bins above its first bin.
    const int b0 = nb - 1 - 2 * tid, b1 = nb - 2 - 2 * tid;
    const int c0 = b0 >= 0 ? hist[b0] : 0;
    const int c1 = b1 >= 0 ? hist[b1] : 0;
    int total;
    const int above = block_excl_scan(c0 + c1, warp_tot, total);
    if (b0 >= 0 && above < remaining && above + c0 >= remaining) {
      found_bin = b0;
      found_above = above;
    } else if (b1 >= 0 && above + c0 < remaining && above + c0 + c1 >= remaining) {
      found_bin = b1;
      found_above = above + c0;
    }
    __syncthreads();
    remaining -= found_above;
    prefix |= static_cast<uint32_t>(found_bin) << shift;
    prefix_mask |= static_cast<uint32_t>(nb - 1) << shift;
    __syncthreads();  // found_* is rewritten by the next pass
  }
  const uint32_t thresh = prefix;
  const int take_equal = remaining;  // >= 1

  // ---- ordered output pass
  int out_base = 0, eq_base = 0;
  for (int c0 = 0; c0 < len; c0 += kThreads * kItems) {
    const int t0 = c0 + tid * kItems;
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      const int t = t0 + i;
      if (t < len) {
        const uint32_t key = order_key(row[t]);
        gt |= static_cast<uint32_t>(key > thresh) << i;
        eq |= static_cast<uint32_t>(key == thresh) << i;
      }
    }
    int eq_total;
    const int eq_rank = eq_base + block_excl_scan(__popc(eq), warp_tot, eq_total);
    uint32_t take = gt;
    int rank = eq_rank;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
      if ((eq >> i) & 1u) {
        if (rank < take_equal) take |= 1u << i;
        ++rank;
      }
    }
    int take_total;
    int pos = out_base + block_excl_scan(__popc(take), warp_tot, take_total);
#pragma unroll
    for (int i = 0; i < kItems; ++i)
      if ((take >> i) & 1u) out[pos++] = t0 + i;
    eq_base += eq_total;
    out_base += take_total;
  }
  for (int i = want + tid; i < p.topk; i += kThreads) out[i] = -1;
}

}  // namespace

cudaError_t launch_select_topk(const TopkParams& p, cudaStream_t stream) {
  select_topk_kernel<<<p.rows, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
