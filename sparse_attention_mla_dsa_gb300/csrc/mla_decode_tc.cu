// mla_decode_tc.cu -- S3 on the 5th-generation tensor cores: absorbed NoPE
// MLA gather-attend with tcgen05 MMAs, accumulators in TMEM.
//
// "glm5next_dsa/layer.rs": module header trap 4 (Q arrives absorbed into the
// 512-wide latent space), attend_rows (one launch for all rows, each with its
// own selection row, seq_len and block-table row; K and V are the same latent
// pool), decode_k (slot = block * block_size + pos % block_size).  Per row and
// head:  z_j = sm_scale * kv_scale * (Q . e4m3(latent_j)),  p = softmax(z),
//        out = kv_scale * sum_j p_j e4m3(latent_j),  lse = log sum_j exp(z_j).
//
// A row's selection is cut into n splits of at most 128 entries (n is a
// function of topk alone); each CTA (8 warps) handles one split of one
// (row, 64-head group):
//   1. gathers its <= 128 selected latent rows (16-byte loads) and widens FP8
//      to f16 (exact) into a 128 x 512 tile in the 128-byte-swizzled layout;
//      loads Q (64 heads, each scaled by a power of two so its bf16 values are
//      exact in f16) as a 64 x 512 K-major operand;
//   2. S^T = Khat Q^T: one thread issues 32 tcgen05.mma (M=128 tokens, N=64
//      heads, K=16 each) into TMEM;
//   3. softmax over the tile's tokens per head, exact (the whole split is in
//      the tile), P^T written as a 64 x 128 K-major f16 operand;
//   4. O^T = V^T P^T: V^T is the same latent tile read as an MN-major operand
//      (dims contiguous), 4 x 8 tcgen05.mma (M=128 dims, N=64 heads, K=16);
//   5. the split's unnormalised O rows and its (max, sum) go to the workspace
//      (staged through shared memory, 16-byte coalesced stores, L2-resident).
// A merge kernel, chained by programmatic dependent launch, combines the n
// splits of every (row, head) in fixed split order and discards the L2 lines
// it consumed, so the partials never reach HBM.
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHeads = 64;             // heads per CTA (MMA N)
constexpr int kTok = 128;              // tokens per split (MMA M of S^T)
constexpr int kMergeThreads = 128;     // merge kernel: one CTA per (row, head), 4 dims per thread
constexpr uint32_t kTileBytes = kTok * 512 * 2;        // latent tile, f16: 8 sub-tiles of 16 KB
constexpr uint32_t kSubTok = kTok * 128;               // one 64-dim sub-tile of the latent tile
constexpr uint32_t kQBytes = kHeads * 512 * 2;         // Q operand, f16: 8 sub-tiles of 8 KB
constexpr uint32_t kSubQ = kHeads * 128;
constexpr uint32_t kPBytes = kHeads * kTok * 2;        // P^T operand: 2 sub-tiles of 8 KB
constexpr uint32_t kSubP = kHeads * 128;
constexpr uint32_t kTmemCols = 512;                    // S^T: cols 0..63, O^T blocks: 64 + 64*mb
constexpr uint64_t kWaitNs = 500ull * 1000ull * 1000ull;

struct __align__(8) Ctl {
  uint64_t bar_s, bar_o;
  uint32_t tmem_base;
  int abort_flag;
  int64_t slot[kTok];
  float qexp[kHeads];  // per-head logit scale
};
constexpr uint32_t kCtlOff = kTileBytes + kQBytes + kPBytes;
constexpr uint32_t kSmemBytes = kCtlOff + sizeof(Ctl) + 1024;  // + alignment slack

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t out;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(codes));
  return out;
}
// Byte offset of 16-byte chunk `c` (0..7) of row `row` inside a 128-byte
// swizzled sub-tile (1024-byte aligned): chunks of 8 rows are XOR-permuted.
__device__ __forceinline__ uint32_t sw128(int row, int c) {
  return static_cast<uint32_t>(row) * 128u + static_cast<uint32_t>((c ^ (row & 7)) * 16);
}
// Descriptor of an MN-major operand in the 128-byte swizzled layout: 64
// contiguous MN elements per 128-byte row, K rows 128 B apart; the next 64 MN
// elements lie `lbo` bytes on, the next 8 K rows 1024 bytes on.
__device__ __forceinline__ uint64_t umma_desc_sw128_mnmajor(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// kind::f16 instruction descriptor: f16 A and B, f32 D, A optionally MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, bool a_mn_major) {
  return (1u << 4) | (a_mn_major ? (1u << 15) : 0u) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
// Drop a 128-byte L2 line without writing it back (its contents become
// undefined); used on partials that have been consumed.
__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
// 32 consecutive TMEM columns of this thread's lane (waited in the same asm).
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_tc_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tile = smem;                 // Khat, f16, [128 tok] x [512 dims], 8 sub-tiles
  uint8_t* qop = smem + kTileBytes;     // Q, f16, [64 heads] x [512 dims], 8 sub-tiles
  uint8_t* pop = qop + kQBytes;         // P^T, f16, [64 heads] x [128 tok], 2 sub-tiles
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);
  float* sm_s = reinterpret_cast<float*>(qop);     // logits [64 heads][128 tok] after S^T

  const int hg = blockIdx.y, r = blockIdx.z;
  const int split = blockIdx.x;
  const int nsplit = p.splits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = split * p.split_len;
  const int nj = max(0, min(p.split_len, p.topk - j0));
  const bool report = hg == 0;
  const int head0 = hg * kHeads;
  const int nheads = min(kHeads, p.heads - head0);

  grid_dep_launch();
  int len = p.rows.seq_lens[r];
  if (len < 0) {
    if (report && split == 0 && tid == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }

  // ---- set-up: barriers, TMEM, slots of this split's entries
  if (tid == 0) {
    mbar_init(&ctl->bar_s, 1);
    mbar_init(&ctl->bar_o, 1);
    fence_mbar_init();
    ctl->abort_flag = 0;
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // ---- Q operand: 4 threads per head, 128 elements each; power-of-two scale
  // per head so every bf16 value is exact in f16.  Heads past the row's count
  // are zero.
  // (Q loads are issued first: they do not depend on the slot lookups.)
  const int qh = tid >> 2, qq = tid & 3;
  uint4 qraw[16];
  {
    const int h = qh, q = qq;
    const bool real = h < nheads;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (static_cast<int64_t>(r) * p.heads + head0 + h) * 512 + q * 128);
#pragma unroll
    for (int j = 0; j < 16; ++j) qraw[j] = real ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
  }
  grid_dep_wait();  // the selection comes from the kernel before
  if (tid < kTok) {
    int64_t slot = -1;
    if (tid < nj) {
      const int idx = __ldg(p.sel + static_cast<int64_t>(r) * p.topk + j0 + tid);
      if (idx != -1) {
        if (idx < 0 || idx >= len) {
          if (report) record_error(p.err, DSA_DEVERR_SELECT, r);
        } else {
          const int32_t* bt = p.rows.block_table + static_cast<int64_t>(r) * p.rows.bt_stride;
          const int bs = p.rows.block_size;
          const int blk = idx / bs;
          const int phys = blk < p.rows.max_blocks_per_seq ? __ldg(bt + blk) : -1;
          const int64_t s = static_cast<int64_t>(phys) * bs + idx % bs;
          if (phys < 0 || s >= p.nslots) {
            if (report) record_error(p.err, DSA_DEVERR_BLOCK, r);
          } else {
            slot = s;
          }
        }
      }
    }
    ctl->slot[tid] = slot;
  }

  {
    const int h = qh, q = qq;
    const uint4* raw = qraw;
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    int e = 0;
    if (amax > 0.0f) frexpf(amax, &e);  // amax < 2^e
    const int sh = max(-100, min(100, 14 - e));
    const float scale = ldexpf(1.0f, sh);
    // Logit scale of this head: sm_scale * kv_scale * log2(e) / 2^sh.
    if (q == 0)
      ctl->qexp[h] = p.sm_scale * p.kv_scale * 1.4426950408889634f * ldexpf(1.0f, -sh);
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // 8 elements = one 16-byte chunk of the operand
      const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
      uint32_t o4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o4[i] = pack_f16x2(__uint_as_float(w[i] << 16) * scale,
                           __uint_as_float(w[i] & 0xFFFF0000u) * scale);
      const int d0 = q * 128 + j * 8;  // first of the 8 dims
      *reinterpret_cast<uint4*>(qop + (d0 >> 6) * kSubQ + sw128(h, (d0 & 63) >> 3)) =
          make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
  __syncthreads();  // slots visible

  // ---- latent tile: 128 tokens x 32 chunks of 16 B, 16 chunks per thread
  {
    uint4 raw[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = tid + j * kThreads;
      const int tok = c >> 5, k = c & 31;
      const int64_t slot = ctl->slot[tok];
      raw[j] = slot >= 0 ? __ldg(reinterpret_cast<const uint4*>(p.pool + slot * 512) + k)
                         : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = tid + j * kThreads;
      const int tok = c >> 5, k = c & 31;  // dims 16k .. 16k+15
      const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
      uint32_t cv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cv[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] & 0xFFFFu));
        cv[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] >> 16));
      }
      uint8_t* sub = tile + (k >> 2) * kSubTok;
      const int c16 = (k & 3) * 2;
      *reinterpret_cast<uint4*>(sub + sw128(tok, c16)) = make_uint4(cv[0], cv[1], cv[2], cv[3]);
      *reinterpret_cast<uint4*>(sub + sw128(tok, c16 + 1)) = make_uint4(cv[4], cv[5], cv[6], cv[7]);
    }
  }
  fence_proxy_async_smem();  // generic-proxy operand writes -> visible to the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // ---- S^T = Khat Q^T (M = 128 tokens, N = 64 heads, K = 512)
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(kTok, kHeads, false);
    const uint32_t a0 = smem_u32(tile), b0 = smem_u32(qop);
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) {
      const uint32_t a = a0 + (kk >> 2) * kSubTok + (kk & 3) * 32;
      const uint32_t b = b0 + (kk >> 2) * kSubQ + (kk & 3) * 32;
      umma_bf16(tmem, umma_desc_sw128_kmajor(a), umma_desc_sw128_kmajor(b), idesc, kk != 0);
    }
    umma_commit(&ctl->bar_s);
  }

  // ---- softmax over the tile's tokens, per head
  {
    // Warps w and w+4 read TMEM lane quarter w%4 (tokens 32*(w%4) + lane),
    // heads 32*(w/4) .. +31, scale them and store the logits transposed.
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&ctl->bar_s, 0, kWaitNs) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok && lane == 0) {
      record_error(p.err, DSA_DEVERR_TIMEOUT, r);
      ctl->abort_flag = 1;
    }
    tc_fence_after();
    const int tok = (warp & 3) * 32 + lane;
    const int hh = (warp >> 2) * 32;
    float v[32];
    tmem_load32(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + hh, v);
    const bool valid = tok < nj && ctl->slot[tok] >= 0;
    __syncthreads();  // every thread has read Q's region as an MMA operand (bar_s) -> reuse it
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int h = hh + i;
      sm_s[h * kTok + tok] = valid ? v[i] * ctl->qexp[h] : -INFINITY;
    }
  }
  __syncthreads();
  {
    // 4 threads per head, 32 tokens each.
    const int h = tid >> 2, q = tid & 3;
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 t4 = *reinterpret_cast<const float4*>(sm_s + h * kTok + q * 32 + i);
      z[i] = t4.x;
      z[i + 1] = t4.y;
      z[i + 2] = t4.z;
      z[i + 3] = t4.w;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, z[i]);
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      z[i] = mx != -INFINITY ? exp2f(z[i] - mx) : 0.0f;
      sum += z[i];
    }
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
    if (q == 0)
      reinterpret_cast<float2*>(p.part_ml)[((static_cast<int64_t>(r) * gridDim.y + hg) * nsplit + split) *
                                               kHeads + h] = make_float2(mx, sum);
    // P^T row h: tokens q*32 .. q*32+31 = 4 chunks of 8 in sub-tile (q*32)/64.
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int t0 = q * 32 + c * 8;
      uint8_t* sub = pop + (t0 >> 6) * kSubP;
      *reinterpret_cast<uint4*>(sub + sw128(h, (t0 & 63) >> 3)) =
          make_uint4(pack_f16x2(z[c * 8], z[c * 8 + 1]), pack_f16x2(z[c * 8 + 2], z[c * 8 + 3]),
                     pack_f16x2(z[c * 8 + 4], z[c * 8 + 5]), pack_f16x2(z[c * 8 + 6], z[c * 8 + 7]));
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- O^T = V^T P^T (4 blocks of M = 128 dims, N = 64 heads, K = 128 tokens)
  if (tid == 0) {
    const uint32_t idesc = idesc_f16(128, kHeads, true);
    const uint32_t a0 = smem_u32(tile), b0 = smem_u32(pop);
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
      for (int kk = 0; kk < kTok / 16; ++kk) {
        // A: dims 128mb.. (two 64-dim sub-tiles, kSubTok apart), tokens 16kk..
        const uint32_t a = a0 + (2 * mb) * kSubTok + kk * 2048;
        const uint32_t b = b0 + (kk >> 2) * kSubP + (kk & 3) * 32;
        umma_bf16(tmem + 64 + mb * 64, umma_desc_sw128_mnmajor(a, kSubTok),
                  umma_desc_sw128_kmajor(b), idesc, kk != 0);
      }
    }
    umma_commit(&ctl->bar_o);
  }
  {
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&ctl->bar_o, 0, kWaitNs) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok && lane == 0) {
      record_error(p.err, DSA_DEVERR_TIMEOUT, r);
      ctl->abort_flag = 1;
    }
    tc_fence_after();
    // Warp w reads lane quarter w%4 (dims 32*(w%4) + lane of each block) of
    // blocks mb = 2*(w/4), 2*(w/4)+1, all 64 heads, into the free tile region
    // as rows [64 heads][512 dims] (consecutive lanes -> consecutive floats).
    float* stage = reinterpret_cast<float*>(tile);
    const int dl = (warp & 3) * 32 + lane;
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      const int mb = (warp >> 2) * 2 + bb;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[32];
        tmem_load32(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + 64 + mb * 64 + hc * 32,
                    v);
        if (bb == 0 && hc == 0) __syncthreads();  // every thread is past bar_o: the tile is free
#pragma unroll
        for (int i = 0; i < 32; ++i) stage[(hc * 32 + i) * 512 + mb * 128 + dl] = v[i];
      }
    }
    tc_fence_before();
    __syncthreads();
    // This split's partial rows, 16-byte coalesced stores (512 B per thread).
    float4* dst = reinterpret_cast<float4*>(
        p.part_o + ((static_cast<int64_t>(r) * gridDim.y + hg) * nsplit + split) * (kHeads * 512));
    const float4* src = reinterpret_cast<const float4*>(stage);
#pragma unroll 8
    for (int i = tid; i < kHeads * 128; i += kThreads) dst[i] = src[i];
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge of the n splits of one (row, head): 128 threads, 4 dims each, splits
// in fixed order; the consumed partial lines are discarded from L2.
__global__ void __launch_bounds__(kMergeThreads) mla_decode_merge_kernel(const DecodeParams p) {
  const int h = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  const int groups = (p.heads + kHeads - 1) / kHeads;
  const int hg = h / kHeads, hl = h % kHeads;
  const int nsplit = p.splits;
  const int64_t base = (static_cast<int64_t>(r) * groups + hg) * nsplit;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  grid_dep_wait();  // the partials come from the kernel before
  grid_dep_launch();
  float mmax = -INFINITY;
  for (int c = 0; c < nsplit; ++c) mmax = fmaxf(mmax, __ldcg(ml + (base + c) * kHeads + hl).x);
  float lsum = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (mmax != -INFINITY) {
    int c = 0;
    for (; c + 8 <= nsplit; c += 8) {  // eight splits' loads in flight at a time
      float2 mlc[8];
      float4 vc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        mlc[u] = __ldcg(ml + (base + c + u) * kHeads + hl);
        vc[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((base + c + u) * kHeads + hl) * 512) + tid);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float f = exp2f(mlc[u].x - mmax);
        lsum += mlc[u].y * f;
        acc.x += vc[u].x * f;
        acc.y += vc[u].y * f;
        acc.z += vc[u].z * f;
        acc.w += vc[u].w * f;
      }
    }
    for (; c < nsplit; ++c) {
      const float2 mlc = __ldcg(ml + (base + c) * kHeads + hl);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + ((base + c) * kHeads + hl) * 512) + tid);
      const float f = exp2f(mlc.x - mmax);
      lsum += mlc.y * f;
      acc.x += v.x * f;
      acc.y += v.y * f;
      acc.z += v.z * f;
      acc.w += v.w * f;
    }
  }
  const float scale = mmax != -INFINITY ? p.kv_scale / lsum : 0.0f;
  uint2 packed;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed.x) : "f"(acc.y * scale), "f"(acc.x * scale));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed.y) : "f"(acc.w * scale), "f"(acc.z * scale));
  const int64_t head = static_cast<int64_t>(r) * p.heads + h;
  reinterpret_cast<uint2*>(p.out + head * 512)[tid] = packed;
  if (tid == 0 && p.lse != nullptr)
    p.lse[head] = mmax != -INFINITY ? (mmax + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
  // Every lane has used its partial values: drop the consumed 128-byte lines
  // (8 lanes share one) from L2 instead of writing them back.
  __syncwarp();
  if ((tid & 7) == 0)
    for (int c = 0; c < nsplit; ++c)
      discard_l2_line(p.part_o + ((base + c) * kHeads + hl) * 512 + tid * 4);
}

}  // namespace

void plan_mla_decode_tc(DecodeParams& p) {
  int n = (p.topk + kTok - 1) / kTok;
  if (n < 1) n = 1;
  p.splits = n;
  p.split_len = (p.topk + n - 1) / n;
}

size_t mla_decode_tc_workspace_bytes(int32_t rows, int32_t heads, int32_t topk) {
  int n = (topk + kTok - 1) / kTok;
  if (n < 1) n = 1;
  const size_t units = static_cast<size_t>(rows) * ((heads + kHeads - 1) / kHeads) * n * kHeads;
  const size_t o_bytes = (units * 512 * sizeof(float) + 255) & ~static_cast<size_t>(255);
  return o_bytes + units * 2 * sizeof(float);
}

void mla_decode_tc_bind_workspace(DecodeParams& p, void* workspace) {
  const size_t units =
      static_cast<size_t>(p.rows.rows) * ((p.heads + kHeads - 1) / kHeads) * p.splits * kHeads;
  p.part_o = static_cast<float*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       ((units * 512 * sizeof(float) + 255) & ~static_cast<size_t>(255)));
}

cudaError_t launch_mla_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, (p.heads + kHeads - 1) / kHeads, p.rows.rows);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_decode_tc_kernel, p);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(p.heads, p.rows.rows, 1);
  mcfg.blockDim = dim3(kMergeThreads, 1, 1);
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&mcfg, mla_decode_merge_kernel, p);
}

}  // namespace dsa

// ------------------------------------------------------------------------------------------
// Allocation-free gather-attend.
//
// Some callers cannot allocate device memory at the point where they run the
// attend: code that runs while a stream is being captured into a CUDA graph
// (an allocation there would either fail or be baked into the graph), code
// whose device memory is owned by another allocator that it may not call, and
// serving loops that must not pay cudaMalloc's implicit device synchronisation
// on the decode path.  This entry point runs the same kernel as
// dsa_mla_decode_fp8 with the split partials in this file-scope device array
// instead of a caller-provided workspace.  The array is
// DSA_NOALLOC_SCRATCH_BYTES long and every GPU that loads the library keeps it
// until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[64] = {};
}  // namespace

extern "C" size_t dsa_noalloc_scratch_bytes(int32_t rows, int32_t heads, int32_t topk) {
  if (rows < 1 || heads < 1 || topk < 1) return 0;
  return dsa::mla_decode_tc_workspace_bytes(rows, heads, topk);
}

extern "C" dsa_status dsa_mla_decode_fp8_noalloc(const dsa_rows* rows, const uint16_t* q,
                                                 const uint8_t* pool, int64_t nslots,
                                                 const int32_t* sel, int32_t topk, int32_t heads,
                                                 int32_t latent_dim, float kv_scale,
                                                 float sm_scale, uint16_t* out,
                                                 float* lse_or_null, void* stream) {
  if (rows == nullptr || rows->rows < 1 || heads < 1 || topk < 1) return DSA_ERR_INVALID_ARG;
  if (dsa_noalloc_scratch_bytes(rows->rows, heads, topk) > DSA_NOALLOC_SCRATCH_BYTES)
    return DSA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSA_ERR_CUDA;
  void* scratch = nullptr;
  {
    // Host code cannot take the array's address directly (its name is a host
    // stand-in); ask the runtime once per device, with that device current.
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
        return DSA_ERR_CUDA;
      g_noalloc_addr[dev] = addr;
    }
    scratch = g_noalloc_addr[dev];
  }
  return dsa_mla_decode_fp8(rows, q, pool, nslots, sel, topk, heads, latent_dim, kv_scale,
                            sm_scale, out, lse_or_null, scratch, DSA_NOALLOC_SCRATCH_BYTES,
                            stream);
}
