// select_topk.cu -- S2: per-row top-k of the indexer scores.
//
// "glm5next_dsa/layer.rs", notes on batch_select_enabled / select_rows_batched:
// the selection is taken under a total order (score DESC, then index ASC), so
// the top-k set is unique; each row's result is a function of its own scores.
//
// One thread-block cluster of C CTAs per row (512 threads each, two CTAs per
// SM; C = 1 up to 4k tokens, at most 8).  CTA c keeps tokens [c*S, (c+1)*S) of the row in
// shared memory as order-preserving 32-bit keys, read from global once.  A
// four-digit radix select (8 bits per digit) finds the key T of the k-th
// largest token, stopping early once every key left in the threshold bin is
// needed.  Scores bunch into few high-order bins, so every histogram
// keeps one counter per (bin, lane): the 32 lanes of a warp never add to the
// same address.  With C > 1 the per-CTA bin totals are summed through
// distributed shared memory and every CTA takes the same decision.  The
// output pass writes every token with key > T plus the lowest-index tokens
// with key == T in ascending token order: slices are in index order, so a
// prefix of the per-CTA counts over the cluster gives each CTA its output
// offset and its share of the tied tokens, and block-wide prefix sums order
// the writes inside it.
//
// The cluster size follows the row length (about 4k keys per CTA).  When the
// launch would then need more CTAs than there are SMs, the cluster is cut to
// one CTA per SM if the longer slices still fit in shared memory (32 rows of
// 64k or 128k: four CTAs each), else to what one wave of two CTAs per SM
// holds if the slices fit two per SM, down to one CTA per row (many short
// rows: a prefill).  The selection is exact, so the cluster size never
// changes a result.
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;             // 8-bit digits
constexpr int kItems = 8;              // consecutive tokens per thread in the output pass
constexpr int kKeysPerCta = 4096;      // target keys per CTA when choosing the cluster size
constexpr int kFastChunks = 4;         // output chunks a slice may have for the count-free path
constexpr size_t kTwoPerSmBytes = 112 * 1024;  // shared memory that leaves room for two CTAs per SM
constexpr size_t kOnePerSmBytes = 227 * 1024;  // the most one CTA may have


__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// Volatile (kept after the cluster barrier) without a memory clobber, so
// consecutive remote loads are issued back to back.
__device__ __forceinline__ int ld_remote_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ int2 ld_remote_s32x2(uint32_t addr) {
  int2 v;
  asm volatile("ld.shared::cluster.v2.s32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
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
    int s = lane < kWarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) warp_tot[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp ? warp_tot[warp - 1] : 0;
  total = warp_tot[kWarps - 1];
  __syncthreads();  // warp_tot may be reused right after
  return before + x - v;
}

// The keys follow this block in shared memory and are read as 16-byte
// vectors: its size must stay a multiple of 16.
struct alignas(16) TopkShared {
  int hist[kBins * 32];          // [bin][lane] counters of the current pass
  int bin_tot[4][kBins];         // per-pass bin totals of this CTA (read remotely)
  int scan_tmp[2 * kBins];       // per-bin exclusive prefix and count of the current pass
  alignas(8) int counts[2];      // this CTA's (key > T, key == T) counts
  alignas(16) int warp_tot[kWarps];
  int found_bin, found_above, found_count;
};
static_assert(sizeof(TopkShared) % 16 == 0, "keys must start 16-byte aligned");

__global__ void __launch_bounds__(kThreads, 2) select_topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkShared& sh = *reinterpret_cast<TopkShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkShared));
  const int r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t crank = cluster_rank();
  const int C = p.cluster;
  grid_dep_wait();  // the scores come from the kernel before
  grid_dep_launch();

  int len = p.seq_lens[r];
  if (len < 0 || len > p.max_len) {
    if (tid == 0 && crank == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }
  int32_t* out = p.sel + static_cast<int64_t>(r) * p.topk;
  const int want = min(p.topk, len);
  if (len <= p.topk) {  // everything visible is selected (uniform over the cluster)
    for (int i = crank * kThreads + tid; i < p.topk; i += C * kThreads) out[i] = i < len ? i : -1;
    return;
  }

  // This CTA's slice of the row, as keys in shared memory.
  const int per = (len + C - 1) / C;
  const int lo = min(len, static_cast<int>(crank) * per);
  const int n = min(len, lo + per) - lo;
  const float* row = p.scores + static_cast<int64_t>(r) * p.max_len + lo;
  // The first pass's histogram (the keys' top 8 bits) is counted as the keys
  // arrive; each later pass's counters are cleared by the threads that read
  // them for the bin totals.
#pragma unroll
  for (int j = 0; j < kBins * 32 / kThreads; ++j) sh.hist[tid + j * kThreads] = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 8 * kThreads) {  // eight loads in flight per thread
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = base + j * kThreads + tid;
      v[j] = i < n ? row[i] : 0.0f;  // plain load: stays after the wait
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = base + j * kThreads + tid;
      if (i < n) {
        const uint32_t key = order_key(v[j]);
        keys[i] = key;
        atomicAdd(&sh.hist[(key >> 24) * 32 + lane], 1);
      }
    }
  }

  // ---- radix select, 8 bits per pass from the top
  uint32_t prefix = 0, prefix_mask = 0;
  int remaining = want;
  bool all_taken = false;  // (uniform) every key equal to the threshold prefix is taken
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (pass > 0) {
#pragma unroll 8
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        if ((key & prefix_mask) == prefix) atomicAdd(&sh.hist[((key >> shift) & 255u) * 32 + lane], 1);
      }
    }
    __syncthreads();
    // Bin totals: 2 threads per bin, 16 lane counters each.  The 16 threads
    // of a warp that share a half start at different counters (rotation by
    // the bin), so each load of the warp touches 32 distinct banks.
    {
      const int b = tid >> 1, q = tid & 1;
      int t = 0;
#pragma unroll
      for (int l = 0; l < 16; ++l) {
        int* h = &sh.hist[b * 32 + q * 16 + ((l + b) & 15)];
        t += *h;
        *h = 0;  // ready for the next pass
      }
      t += __shfl_xor_sync(0xFFFFFFFFu, t, 1);
      if (q == 0) sh.bin_tot[pass][b] = t;
    }
    if (C > 1) cluster_sync();  // every CTA's totals of this pass are visible
    else __syncthreads();
    // Warp w < 8 scans bins 255-32w .. 224-32w (descending order of bins).
    if (warp < kBins / 32) {
      const int b = kBins - 1 - (warp * 32 + lane);
      int c = 0;
      if (C > 1) {
        int v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < C) v[k] = ld_remote_s32(remote_addr(&sh.bin_tot[pass][b], k));
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (k < C) c += v[k];
      } else {
        c = sh.bin_tot[pass][b];
      }
      int x = c;  // inclusive scan within the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      sh.warp_tot[warp] = 0;  // placeholder, overwritten below
      __syncwarp();
      if (lane == 31) sh.warp_tot[warp] = x;
      sh.scan_tmp[warp * 32 + lane] = x - c;   // exclusive within the warp
      sh.scan_tmp[kBins + warp * 32 + lane] = c;
    }
    __syncthreads();
    if (warp < kBins / 32) {
      // Totals of the scanning warps before this one (two vector loads).
      const int4 t0 = *reinterpret_cast<const int4*>(&sh.warp_tot[0]);
      const int4 t1 = *reinterpret_cast<const int4*>(&sh.warp_tot[4]);
      const int before = (warp > 0 ? t0.x : 0) + (warp > 1 ? t0.y : 0) + (warp > 2 ? t0.z : 0) +
                         (warp > 3 ? t0.w : 0) + (warp > 4 ? t1.x : 0) + (warp > 5 ? t1.y : 0) +
                         (warp > 6 ? t1.z : 0);
      const int above = before + sh.scan_tmp[warp * 32 + lane];
      const int c = sh.scan_tmp[kBins + warp * 32 + lane];
      if (above < remaining && above + c >= remaining) {
        sh.found_bin = kBins - 1 - (warp * 32 + lane);
        sh.found_above = above;
        sh.found_count = c;
      }
    }
    __syncthreads();
    remaining -= sh.found_above;
    prefix |= static_cast<uint32_t>(sh.found_bin) << shift;
    prefix_mask |= 255u << shift;
    all_taken = sh.found_count == remaining;
    __syncthreads();  // found_* / hist are rewritten by the next pass
    // Every key in the threshold bin is needed: the selection is the keys
    // whose top bits are >= the prefix found so far, whatever the lower bits.
    if (all_taken) break;
  }
  const uint32_t thresh = prefix;
  const int take_equal = remaining;  // >= 1, counted over the whole row

  // ---- up to kFastChunks output chunks a slice (every CTA of the cluster:
  // the slice length is uniform) with every key at the threshold prefix
  // taken: the output's own scans of the take bits give this CTA's count
  // too, so the count pass and its scan are skipped; the take bits wait in
  // registers for the exchange.  The exchange and the barriers are those of
  // the general path below.
  if (C > 1 && all_taken && per <= kFastChunks * kThreads * kItems) {
    uint32_t take[kFastChunks];
    int pos[kFastChunks];
    int count = 0;
#pragma unroll
    for (int k = 0; k < kFastChunks; ++k) {
      take[k] = 0;
      pos[k] = 0;
      const int c0 = k * kThreads * kItems;
      if (c0 < n) {  // (uniform over the CTA)
        const int t0 = c0 + tid * kItems;
        uint32_t kv[kItems];
        if (t0 + kItems <= n) {
          const uint4 u0 = *reinterpret_cast<const uint4*>(keys + t0);
          const uint4 u1 = *reinterpret_cast<const uint4*>(keys + t0 + 4);
          kv[0] = u0.x; kv[1] = u0.y; kv[2] = u0.z; kv[3] = u0.w;
          kv[4] = u1.x; kv[5] = u1.y; kv[6] = u1.z; kv[7] = u1.w;
        } else {
#pragma unroll
          for (int i = 0; i < kItems; ++i) kv[i] = t0 + i < n ? keys[t0 + i] : 0u;
        }
#pragma unroll
        for (int i = 0; i < kItems; ++i)
          if (t0 + i < n) take[k] |= static_cast<uint32_t>((kv[i] & prefix_mask) >= thresh) << i;
        int chunk_total;
        pos[k] = count + block_excl_scan(__popc(take[k]), sh.warp_tot, chunk_total);
        count += chunk_total;
      }
    }
    if (tid == 0) {
      sh.counts[0] = count;
      sh.counts[1] = 0;
    }
    cluster_sync();
    int2 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c < static_cast<int>(crank)) v[c] = ld_remote_s32x2(remote_addr(&sh.counts[0], c));
    int base = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c < static_cast<int>(crank)) base += v[c].x;
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
#pragma unroll
    for (int k = 0; k < kFastChunks; ++k) {
      int q = base + pos[k];
      const int t0 = k * kThreads * kItems + tid * kItems;
#pragma unroll
      for (int i = 0; i < kItems; ++i)
        if ((take[k] >> i) & 1u) out[q++] = lo + t0 + i;
    }
    for (int i = want + crank * kThreads + tid; i < p.topk; i += C * kThreads) out[i] = -1;
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return;
  }

  // ---- this CTA's counts, then its offsets from the CTAs before it.  When
  // every key at the threshold prefix is taken a key is selected iff its
  // masked bits are >= the prefix (one count, one scan per chunk); otherwise
  // keys above the threshold are taken and the tied ones by rank, lowest index
  // first.
  int out_base = 0, eq_base = 0;
  bool exit_arrived = false;
  if (C > 1) {
    int gt_n = 0, eq_n = 0;
    if (all_taken) {
#pragma unroll 8
      for (int i = tid; i < n; i += kThreads) gt_n += (keys[i] & prefix_mask) >= thresh;
    } else {
#pragma unroll 8
      for (int i = tid; i < n; i += kThreads) {
        const uint32_t key = keys[i];
        gt_n += key > thresh;
        eq_n += key == thresh;
      }
    }
    int gt_total, eq_total = 0;
    block_excl_scan(gt_n, sh.warp_tot, gt_total);
    if (!all_taken) block_excl_scan(eq_n, sh.warp_tot, eq_total);
    if (tid == 0) {
      sh.counts[0] = gt_total;
      sh.counts[1] = eq_total;
    }
    cluster_sync();
    int2 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c < static_cast<int>(crank)) v[c] = ld_remote_s32x2(remote_addr(&sh.counts[0], c));
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c < static_cast<int>(crank)) {
        out_base += v[c].x + min(v[c].y, max(0, take_equal - eq_base));
        eq_base += v[c].y;
      }
    // Last remote read done: arrive now, wait just before leaving, so no CTA
    // exits while another may still read its shared memory.
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    exit_arrived = true;
  }

  // ---- ordered output of this slice
  for (int c0 = 0; c0 < n; c0 += kThreads * kItems) {
    const int t0 = c0 + tid * kItems;
    uint32_t kv[kItems];
    if (t0 + kItems <= n) {  // two 16-byte loads (t0 is a multiple of 8)
      const uint4 u0 = *reinterpret_cast<const uint4*>(keys + t0);
      const uint4 u1 = *reinterpret_cast<const uint4*>(keys + t0 + 4);
      kv[0] = u0.x; kv[1] = u0.y; kv[2] = u0.z; kv[3] = u0.w;
      kv[4] = u1.x; kv[5] = u1.y; kv[6] = u1.z; kv[7] = u1.w;
    } else {
#pragma unroll
      for (int i = 0; i < kItems; ++i) kv[i] = t0 + i < n ? keys[t0 + i] : 0u;
    }
    uint32_t take = 0;
    if (all_taken) {
#pragma unroll
      for (int i = 0; i < kItems; ++i)
        if (t0 + i < n) take |= static_cast<uint32_t>((kv[i] & prefix_mask) >= thresh) << i;
    } else {
      uint32_t eq = 0;
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        if (t0 + i < n) {
          take |= static_cast<uint32_t>(kv[i] > thresh) << i;
          eq |= static_cast<uint32_t>(kv[i] == thresh) << i;
        }
      }
      int chunk_eq;
      int rank = eq_base + block_excl_scan(__popc(eq), sh.warp_tot, chunk_eq);
#pragma unroll
      for (int i = 0; i < kItems; ++i) {
        if ((eq >> i) & 1u) {
          if (rank < take_equal) take |= 1u << i;
          ++rank;
        }
      }
      eq_base += chunk_eq;
    }
    int chunk_take;
    int pos = out_base + block_excl_scan(__popc(take), sh.warp_tot, chunk_take);
#pragma unroll
    for (int i = 0; i < kItems; ++i)
      if ((take >> i) & 1u) out[pos++] = lo + t0 + i;
    out_base += chunk_take;
  }
  for (int i = want + crank * kThreads + tid; i < p.topk; i += C * kThreads) out[i] = -1;
  if (exit_arrived) asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

int topk_cluster_size(int32_t max_len, int32_t rows, int num_sms) {
  int c = (max_len + kKeysPerCta - 1) / kKeysPerCta;
  c = c < 1 ? 1 : (c > 8 ? 8 : c);
  // One CTA per SM first (clusters then pack into the GPCs without a
  // straggler wave; a slice may then take up to a whole SM's shared memory),
  // else two.
  const long long sms = num_sms > 0 ? num_sms : 1;
  for (long long slots = sms; slots <= 2 * sms; slots += sms) {
    if (static_cast<long long>(rows) * c <= slots) break;
    const long long fit = slots / (rows > 0 ? rows : 1);
    const int cut = static_cast<int>(fit < 1 ? 1 : fit);
    if (cut < c && topk_smem_bytes(max_len, cut) <= (slots == sms ? kOnePerSmBytes : kTwoPerSmBytes)) {
      c = cut;
      break;
    }
  }
  return c;
}

size_t topk_smem_bytes(int32_t max_len, int cluster) {
  const size_t per = (static_cast<size_t>(max_len) + cluster - 1) / cluster;
  return sizeof(TopkShared) + per * sizeof(uint32_t);
}

cudaError_t launch_select_topk(const TopkParams& p, cudaStream_t stream) {
  const size_t smem = topk_smem_bytes(p.max_len, p.cluster);
  cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.cluster, p.rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = dependent_launch_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, select_topk_kernel, p);
}

}  // namespace dsa
