// index_scores.cu -- S1: lightning-indexer scores as a TMA-fed tcgen05 MMA
// with the ReLU / head-weight / gate epilogue read straight out of TMEM.
//
// "glm5next_dsa/layer.rs", module header: q_idx (FP32 out of wq_b), k_normed
// and gate (per token, in the indexer cache), and the head weights (already
// carrying index_heads^-0.5, trap 3) feed select_tokens; the score kernel does
// not scale.  Per row r and visible token t:
//     s_r(t) = gate(t) * sum_h w_r[h] * relu(q_r[h] . k(t))
//
// Mapping onto the tensor core ("swap AB": tokens are M):
//   A = 128 keys x D (bf16, K-major, TMA with 128-byte swizzle)
//   B = N x D, N = (rows sharing the sequence) x heads, K-major
//   D = 128 x N FP32 accumulators in TMEM (lane = token, column = row*heads+h)
// q_idx is FP32 on the pages; a single bf16 rounding of q would cost ~1e-3
// relative per head dot, so q = q_hi + q_lo with both halves bf16 and the
// two products accumulate into the same TMEM columns.  Keys are bf16 already,
// so the bytes read are unchanged.
//
// CTA roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues the
// MMAs (one thread), warps 2-5 are the epilogue (one TMEM lane quarter each).
// A CTA handles `chunk_tiles` consecutive 128-token tiles of one launch group
// (at most 64 score columns: rows of a sequence beyond that form further
// groups); the grid is (sub-group, chunk, sequence) and CTAs past a group's
// length exit.
// The arithmetic of every score is the same whichever CTA, chunk or launch
// group computes it, so a row's scores do not depend on the other rows.
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kTileM = 128;
constexpr int kThreads = 192;
constexpr int kMaxStages = 6;
constexpr int kMaxSubRows = 32;

struct __align__(8) IndexCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int max_len_group;
  int row_len[kMaxSubRows];
  int64_t base;
};

__device__ __forceinline__ void set_abort(IndexCtl* c, int* err, int row) {
  record_error(err, DSA_DEVERR_TIMEOUT, row);
  *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}
__device__ __forceinline__ bool aborted(IndexCtl* c) {
  return *reinterpret_cast<volatile int*>(&c->abort_flag) != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    index_scores_kernel(const __grid_constant__ CUtensorMap kmap, const IndexParams p) {
  constexpr int kSub = D / 64;                       // 64-element K sub-tiles per operand
  constexpr uint32_t kStageBytes = kTileM * D * 2;   // one 128 x D bf16 key tile
  constexpr int kKSteps = D / 16;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_launch();

  // ---------------------------------------------------------------- layout
  const int npad = p.npad;
  const uint32_t b_bytes = static_cast<uint32_t>(npad) * D * 2;  // one of hi / lo
  uint8_t* stage_base = smem;
  uint8_t* b_hi = smem + p.stages * kStageBytes;
  uint8_t* b_lo = b_hi + b_bytes;
  float* w_s = reinterpret_cast<float*>(b_lo + b_bytes);
  IndexCtl* ctl = reinterpret_cast<IndexCtl*>(w_s + npad);

  // ---------------------------------------------------------------- launch group
  // Grid (sub-group, chunk, sequence): the sub-groups of a sequence are
  // adjacent in launch order, so they stream the same key tiles together and
  // all but the first read them from L2.
  const int seq = blockIdx.z, sub = blockIdx.x;
  const int seq_row0 = seq * p.rows_per_seq;
  const int r0 = seq_row0 + sub * p.sub_rows;
  const int nrows = min(p.sub_rows, seq_row0 + p.rows_per_seq - r0);
  const int nreal = nrows * p.heads;
  const int t_begin = blockIdx.y * p.chunk_tiles;
  const int stages = p.stages;
  const float* qsrc = p.q_idx + static_cast<int64_t>(r0) * p.heads * D;

  // ---------------------------------------------------------------- before the wait
  // Every input here may be the output of the kernel before (the key arena
  // and gates of an indexer write, q and the head weights of a projection,
  // row metadata written on the device), so nothing is loaded before
  // grid_dep_wait().  What overlaps the kernel before: barrier set-up, the
  // tensor map, and L2 prefetches of this CTA's first key tiles and of its q
  // rows (a prefetch only warms L2, where the device's writes land, so it
  // cannot make a later load return a stale value; the arena base used for
  // the prefetch address may be stale, which only wastes the prefetch).
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], 4);
    }
    mbar_init(&ctl->drain, 1);
    fence_mbar_init();
    tma_prefetch_map(&kmap);
    const int64_t base_hint = *reinterpret_cast<const volatile int64_t*>(p.idx_base + seq_row0);
    for (int i = 0; i < min(stages, p.chunk_tiles); ++i) {
      const int64_t y = base_hint + static_cast<int64_t>(t_begin + i) * kTileM;
      if (y >= 0 && y < p.idx_tokens)
#pragma unroll
        for (int sb = 0; sb < kSub; ++sb) tma_prefetch_l2_2d(&kmap, sb * 64, static_cast<int32_t>(y));
    }
  }
  // B operand: q split into bf16 hi + lo, written in the 128-byte-swizzled
  // K-major layout the MMA descriptor expects (row n at n*128 B inside a
  // 64-element sub-tile, 16-byte chunk c stored at chunk c ^ (n % 8)).
  // Vector v is 8 floats of q row n = v / (D/8); eight vectors per thread are
  // loaded before any is used (one round trip per eight vectors).
  const int vec_per_row = D / 8;
  const int nvec = npad * vec_per_row;
  constexpr int kBatch = 8;
  auto load_batch = [&](int v0, float4 (&u)[kBatch][2]) {
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int v = v0 + k * kThreads;
      const int n = v / vec_per_row, c8 = v % vec_per_row;
      if (v < nvec && n < nreal) {
        const float4* src = reinterpret_cast<const float4*>(qsrc + static_cast<int64_t>(n) * D + c8 * 8);
        u[k][0] = ld_dep_f4(src);
        u[k][1] = ld_dep_f4(src + 1);
      } else {
        u[k][0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        u[k][1] = u[k][0];
      }
    }
  };
  auto convert_vec = [&](int v, const float4& u0, const float4& u1) {
    const int n = v / vec_per_row, c8 = v % vec_per_row;
    const float x[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(x[2 * i]);
      const __nv_bfloat16 h1 = __float2bfloat16_rn(x[2 * i + 1]);
      const float r0f = x[2 * i] - __bfloat162float(h0);
      const float r1f = x[2 * i + 1] - __bfloat162float(h1);
      hi[i] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
      lo[i] = pack_bf16x2(r0f, r1f);
    }
    const int sb = (c8 * 8) / 64, chunk = c8 & 7;
    const uint32_t off = sb * (npad * 128) + n * 128 + ((chunk ^ (n & 7)) * 16);
    *reinterpret_cast<uint4*>(b_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(b_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  };
  auto head_weight = [&](int n) {
    return n < nreal ? *reinterpret_cast<const volatile float*>(p.head_w + static_cast<int64_t>(r0) * p.heads + n)
                     : 0.0f;
  };
  // q and the head weights may come from the kernel before: prefetched into
  // L2 here, loaded and converted after the wait.
  for (int off = threadIdx.x * 32; off < nreal * D; off += kThreads * 32)
    prefetch_l2(qsrc + off);  // 128-byte lines
  if (threadIdx.x < nrows) {
    prefetch_l2(p.seq_lens + r0 + threadIdx.x);
    prefetch_l2(p.idx_base + r0 + threadIdx.x);
  }
  grid_dep_wait();

  // Row lengths and arena bases: one load per row, all rows in parallel.
  if (threadIdx.x < 32) {
    const bool report = blockIdx.y == 0;
    const int j = threadIdx.x;
    const int64_t base = p.idx_base[seq_row0];
    int len = 0;
    if (j < nrows) {
      const int r = r0 + j;
      len = p.seq_lens[r];
      const int64_t rb = p.idx_base[r];
      if (len < 0 || len > p.max_len) {
        if (report) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
        len = 0;
      } else if (rb != base || base < 0 || base + len > p.idx_tokens) {
        if (report) record_error(p.err, DSA_DEVERR_ARENA, r);
        len = 0;
      } else if (p.idx_written != nullptr && len > p.idx_written[seq]) {
        // the sequence's keys stop before this row's range: rows never written
        if (report) record_error(p.err, DSA_DEVERR_BEHIND, r);
        len = 0;
      }
      ctl->row_len[j] = len;
    }
    int maxlen = len;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxlen = max(maxlen, __shfl_xor_sync(0xFFFFFFFFu, maxlen, o));
    if (j == 0) {
      ctl->max_len_group = maxlen;
      ctl->base = base;
      ctl->abort_flag = 0;
    }
  }
  __syncthreads();
  const int tiles = (ctl->max_len_group + kTileM - 1) / kTileM;
  const int t_end = min(t_begin + p.chunk_tiles, tiles);
  if (t_begin >= t_end) return;  // uniform across the CTA, before any TMA, MMA or TMEM use
  const int ntiles = t_end - t_begin;
  const int64_t base = ctl->base;

  // ---------------------------------------------------------------- setup
  uint64_t policy = 0;
  int issued = 0;
  if (threadIdx.x == 0) {
    policy = l2_policy_evict_first();
    // The first `stages` tiles need no empty-slot wait.
    for (; issued < min(stages, ntiles); ++issued) {
      uint8_t* dst = stage_base + issued * kStageBytes;
      const int32_t y = static_cast<int32_t>(base + static_cast<int64_t>(t_begin + issued) * kTileM);
      mbar_arrive_expect_tx(&ctl->full[issued], kStageBytes);
#pragma unroll
      for (int sb = 0; sb < kSub; ++sb)
        tma_load_2d(dst + sb * (kTileM * 128), &kmap, &ctl->full[issued], sb * 64, y, policy);
    }
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, p.tmem_cols);
    tmem_relinquish();
  }
  {
    float4 u[kBatch][2];
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kBatch * kThreads) {
      load_batch(v0, u);
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int v = v0 + k * kThreads;
        if (v < nvec) convert_vec(v, u[k][0], u[k][1]);
      }
    }
    for (int n = threadIdx.x; n < npad; n += kThreads) w_s[n] = head_weight(n);
  }
  fence_proxy_async_smem();  // generic-proxy smem writes -> visible to the MMA
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  // ---------------------------------------------------------------- roles
  if (warp == 0) {
    if (lane == 0) {
      for (; issued < ntiles; ++issued) {
        if (aborted(ctl)) break;
        const int s = issued % stages;
        const uint32_t use = issued / stages;
        if (!mbar_wait(&ctl->empty[s], (use - 1) & 1, p.wait_ns)) {
          set_abort(ctl, p.err, r0);
          break;
        }
        uint8_t* dst = stage_base + s * kStageBytes;
        const int32_t y = static_cast<int32_t>(base + static_cast<int64_t>(t_begin + issued) * kTileM);
        mbar_arrive_expect_tx(&ctl->full[s], kStageBytes);
#pragma unroll
        for (int sb = 0; sb < kSub; ++sb)
          tma_load_2d(dst + sb * (kTileM * 128), &kmap, &ctl->full[s], sb * 64, y, policy);
      }
      // Never leave with a copy in flight: wait (bounded) for the last loads.
      for (int i = max(0, issued - stages); i < issued; ++i)
        mbar_wait(&ctl->full[i % stages], (i / stages) & 1, kDrainWaitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTileM, npad);
      const uint32_t a0 = smem_u32(stage_base), bh = smem_u32(b_hi), bl = smem_u32(b_lo);
      for (int i = 0; i < ntiles; ++i) {
        if (aborted(ctl)) break;
        const int s = i % stages, a = i & 1;
        if (!mbar_wait(&ctl->full[s], (i / stages) & 1, p.wait_ns)) {
          set_abort(ctl, p.err, r0);
          break;
        }
        if (i >= 2 && !mbar_wait(&ctl->tempty[a], ((i >> 1) - 1) & 1, p.wait_ns)) {
          set_abort(ctl, p.err, r0);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + a * npad;
        const uint32_t a_stage = a0 + s * kStageBytes;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t b_base = half ? bl : bh;
#pragma unroll
          for (int kk = 0; kk < kKSteps; ++kk) {
            const uint32_t a_addr = a_stage + (kk >> 2) * (kTileM * 128) + (kk & 3) * 32;
            const uint32_t b_addr = b_base + (kk >> 2) * (npad * 128) + (kk & 3) * 32;
            umma_bf16(d_tmem, umma_desc_sw128_kmajor(a_addr), umma_desc_sw128_kmajor(b_addr),
                      idesc, (half | kk) != 0);
          }
        }
        umma_commit(&ctl->empty[s]);
        umma_commit(&ctl->tfull[a]);
      }
      // Every MMA issued by this thread is complete before TMEM is released.
      umma_commit(&ctl->drain);
      mbar_wait(&ctl->drain, 0, kDrainWaitNs);
    }
  } else {
    // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. those tokens.
    const int quarter = warp & 3;
    const int lane_tok = quarter * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const int heads = p.heads;
    const int cols_per_row = (heads % 16 == 0) ? heads : npad;  // heads%16 != 0 -> one row
    // Each tile's gate is loaded one tile ahead, so the load's DRAM latency
    // hides behind the TMA and the MMAs (plain loads: the gates may come from
    // the kernel before, which the wait at the top has ordered).
    const int max_len_group = ctl->max_len_group;
    auto load_gate = [&](int i) {
      const int t = (t_begin + i) * kTileM + lane_tok;
      return (i < ntiles && t < max_len_group) ? p.gate[base + t] : static_cast<uint16_t>(0);
    };
    uint16_t g_next = load_gate(0);
    for (int i = 0; i < ntiles; ++i) {
      if (__shfl_sync(0xFFFFFFFFu, aborted(ctl) ? 1 : 0, 0)) break;
      const int a = i & 1;
      const int t = (t_begin + i) * kTileM + lane_tok;
      const float g = __bfloat162float(__ushort_as_bfloat16(g_next));
      g_next = load_gate(i + 1);
      // One lane polls; the warp then continues together (tcgen05.ld is
      // warp-collective), ordered after the wait by the warp sync + fence.
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&ctl->tfull[a], (i >> 1) & 1, p.wait_ns) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) set_abort(ctl, p.err, r0);
        break;
      }
      tc_fence_after();
      const uint32_t acc = lane_addr + a * npad;
      for (int j = 0; j < nrows; ++j) {
        float sum = 0.0f;
        const int c_begin = j * cols_per_row;
        for (int c0 = c_begin; c0 < c_begin + cols_per_row; c0 += 16) {
          float v[16];
          tmem_load16(acc + c0, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int n = c0 + k;
            if (n < nreal) sum = fmaf(w_s[n], fmaxf(v[k], 0.0f), sum);
          }
        }
        if (t < ctl->row_len[j])
          p.scores[static_cast<int64_t>(r0 + j) * p.max_len + t] = g * sum;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tempty[a]);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace

void plan_index_scores(IndexParams& p, int num_sms) {
  const int64_t tiles_max = (static_cast<int64_t>(p.max_len) + kTileM - 1) / kTileM;
  const int64_t groups = static_cast<int64_t>(p.rows / p.rows_per_seq) * p.subs_per_seq;
  const int64_t upper = tiles_max * groups;
  int64_t chunk = (upper + 16LL * num_sms - 1) / (16LL * num_sms);
  // Each CTA builds its q hi/lo operand (npad x D) before streaming keys: on
  // large launches give it at least npad/8 tiles so that build stays small
  // next to the key bytes it serves.
  if (upper >= 8LL * num_sms) chunk = chunk > p.npad / 8 ? chunk : p.npad / 8;
  chunk = chunk < 1 ? 1 : (chunk > 16 ? 16 : chunk);
  p.chunk_tiles = static_cast<int32_t>(chunk);

  const uint32_t stage_bytes = kTileM * p.dim * 2;
  const uint32_t b_bytes = 2u * p.npad * p.dim * 2;
  const uint32_t fixed = b_bytes + p.npad * 4 + sizeof(IndexCtl) + 1024;  // + alignment slack
  const uint32_t two_per_sm = 113u * 1024u, one_per_sm = 226u * 1024u;
  int stages = 0;
  if (fixed + 2 * stage_bytes <= two_per_sm)
    stages = static_cast<int>((two_per_sm - fixed) / stage_bytes);
  else
    stages = static_cast<int>((one_per_sm - fixed) / stage_bytes);
  stages = stages > 4 ? 4 : stages;
  if (stages > chunk) stages = static_cast<int>(chunk);
  if (stages < 1) stages = 1;
  p.stages = stages;
  p.smem_bytes = fixed + stages * stage_bytes;

  uint32_t cols = 32;
  while (cols < 2u * p.npad) cols <<= 1;
  p.tmem_cols = cols;
}

cudaError_t launch_index_scores(const IndexParams& p, const CUtensorMap& kmap,
                                cudaStream_t stream) {
  const int64_t tiles_max = (static_cast<int64_t>(p.max_len) + kTileM - 1) / kTileM;
  const int64_t chunks = (tiles_max + p.chunk_tiles - 1) / p.chunk_tiles;
  const int64_t groups = static_cast<int64_t>(p.rows / p.rows_per_seq) * p.subs_per_seq;
  if (chunks <= 0 || groups <= 0) return cudaSuccess;
  const int64_t seqs = p.rows / p.rows_per_seq;
  if (chunks > 65535 || seqs > 65535 || p.subs_per_seq > 65535)
    return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(p.subs_per_seq), static_cast<unsigned>(chunks),
            static_cast<unsigned>(seqs));
  cudaError_t e;
  auto kernel = p.dim == 64 ? index_scores_kernel<64> : index_scores_kernel<128>;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, kmap, p);
}

}  // namespace dsa
