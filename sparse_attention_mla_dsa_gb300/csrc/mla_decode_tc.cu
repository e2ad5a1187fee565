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
// A row's selection is cut into n splits of at most 256 entries (512 when the
// row has more than 64 heads); n and the split length depend on topk and the
// head count only, never on the number of rows, so a row's arithmetic is the
// same in any launch.  Each CTA (8 warps) runs one split of one (row, 64-head
// group) as a loop over 128-entry tiles, with an online softmax:
//   0. resolves the slots of all its entries once, loads Q (64 heads, each
//      scaled by a power of two so its bf16 values are exact in f16) as a
//      64 x 512 K-major operand that stays resident;
//   1. widens the tile's FP8 latent rows (already in registers) to f16
//      (exact) into a 128 x 512 tile in the 128-byte-swizzled layout, then
//      issues the 16-byte gathers of the next tile into the same registers,
//      so their latency hides behind this tile's MMAs and softmax;
//   2. S^T = Khat Q^T: one thread issues 32 tcgen05.mma (M=128 tokens, N=64
//      heads, K=16 each) into TMEM;
//   3. softmax: each thread holds one token's logits for 32 heads; per-head
//      tile maxima come from a butterfly transpose-reduction across the warp
//      and a 4-way exchange in shared memory.  The running maximum of a head
//      only moves when a tile exceeds it by more than 2^8 (then the head's
//      accumulated O columns and sum are rescaled in place); otherwise the
//      stale maximum is kept, so the weights stay below 2^8 and exact math
//      is unchanged.  P^T is written as a 128 x 64 MN-major f16 operand;
//   4. O^T += V^T P^T: V^T is the same latent tile read as an MN-major
//      operand (dims contiguous), 4 x 8 tcgen05.mma (M=128 dims, N=64 heads,
//      K=16) accumulating in TMEM across the split's tiles;
//   5. with one split the CTA normalises and writes the bf16 output (and
//      lse) itself; otherwise the split's unnormalised O rows and its (max,
//      sum) go to the workspace (staged through shared memory, 16-byte
//      coalesced stores, L2-resident) and a merge kernel, chained by
//      programmatic dependent launch, combines the n splits of every (row,
//      head) in fixed split order and discards the L2 lines it consumed.
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHeads = 64;             // heads per CTA (MMA N)
constexpr int kTok = 128;              // entries per tile (MMA M of S^T)
constexpr int kMaxTiles = 4;           // tiles per split
constexpr int kMergeThreads = 128;     // merge kernel: one CTA per (row, head), 4 dims per thread
constexpr float kRescaleLog2 = 8.0f;   // a head's running max moves only past this margin
constexpr uint32_t kTileBytes = kTok * 512 * 2;        // latent tile, f16: 8 sub-tiles of 16 KB
constexpr uint32_t kSubTok = kTok * 128;               // one 64-dim sub-tile of the latent tile
constexpr uint32_t kQBytes = kHeads * 512 * 2;         // Q operand, f16: 8 sub-tiles of 8 KB
constexpr uint32_t kSubQ = kHeads * 128;
constexpr uint32_t kPBytes = kTok * kHeads * 2;        // P^T operand, MN-major: 128 rows of 128 B
constexpr uint32_t kTmemCols = 512;                    // S^T: cols 0..63, O^T blocks: 64 + 64*mb
constexpr uint64_t kWaitNs = 500ull * 1000ull * 1000ull;

struct __align__(16) Ctl {
  uint64_t bar_s, bar_o;
  uint32_t tmem_base;
  int pad[3];
  alignas(16) float qexp[kHeads];   // per-head logit scale
  alignas(16) float red[4][kHeads]; // per lane quarter: head maxima, then sums
  float lfin[kHeads];               // final per-head sums and maxima
  float mfin[kHeads];
  int32_t slot[kMaxTiles * kTok];   // -1: no latent row
};
constexpr uint32_t kCtlOff = kTileBytes + kQBytes + kPBytes;
constexpr uint32_t kSmemBytes = kCtlOff + sizeof(Ctl) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

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
// kind::f16 instruction descriptor: f16 A and B, f32 D; A and B each K-major
// or MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (a_mn_major ? (1u << 15) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
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
// The same columns written back from registers (the caller waits with
// tmem_store_wait before the values are used by an MMA).
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One butterfly step of a warp transpose-reduction: on entry v[0..2S) are
// values of 2S heads in this lane; on exit v[0..S) hold, for the S heads
// selected by lane bit S, the reduction over this lane and lane ^ S.  After
// the steps S = 16, 8, 4, 2, 1, v[0] of lane l is the reduction of head l over
// the 32 lanes, in an order fixed by the lane numbering.
template <int S, bool kMax>
__device__ __forceinline__ void butterfly_step(float* v, int lane) {
  const bool up = (lane & S) != 0;
#pragma unroll
  for (int j = 0; j < S; ++j) {
    const float send = up ? v[j] : v[j + S];
    const float keep = up ? v[j + S] : v[j];
    const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, S);
    v[j] = kMax ? fmaxf(keep, recv) : keep + recv;
  }
}
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane) {
  butterfly_step<16, kMax>(v, lane);
  butterfly_step<8, kMax>(v, lane);
  butterfly_step<4, kMax>(v, lane);
  butterfly_step<2, kMax>(v, lane);
  butterfly_step<1, kMax>(v, lane);
  return v[0];
}

// Bounded wait of a whole warp on an mbarrier phase; a timeout is recorded
// once and later waits of this warp are skipped.
__device__ __forceinline__ void warp_wait(uint64_t* bar, uint32_t parity, bool& alive, int lane,
                                          int* err, int r) {
  int ok = 1;
  if (alive) {
    if (lane == 0) ok = mbar_wait(bar, parity, kWaitNs) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  }
  if (alive && !ok) {
    if (lane == 0) record_error(err, DSA_DEVERR_TIMEOUT, r);
    alive = false;
  }
}

// 16-byte gathers of one tile: warp w loads the latent rows of tokens
// w, w+8, ..., w+120 of the tile, lane l their bytes 16l..16l+15.
__device__ __forceinline__ void gather_tile(uint4 (&raw)[16], const int32_t* slot,
                                            const uint8_t* pool, int e0, int nj, int warp,
                                            int lane) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int e = e0 + warp + 8 * j;
    const int s = e < nj ? slot[e] : -1;
    raw[j] = s >= 0 ? __ldg(reinterpret_cast<const uint4*>(pool + static_cast<int64_t>(s) * 512) + lane)
                    : make_uint4(0, 0, 0, 0);
  }
}
// The same rows widened to f16 into the latent tile (token = row, dims
// 16l..16l+15 = two 16-byte chunks of sub-tile l/4).
__device__ __forceinline__ void store_tile(uint8_t* tile, const uint4 (&raw)[16], int warp,
                                           int lane) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int tok = warp + 8 * j;
    const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
    uint32_t cv[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cv[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] & 0xFFFFu));
      cv[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] >> 16));
    }
    uint8_t* sub = tile + (lane >> 2) * kSubTok;
    const int c16 = (lane & 3) * 2;
    *reinterpret_cast<uint4*>(sub + sw128(tok, c16)) = make_uint4(cv[0], cv[1], cv[2], cv[3]);
    *reinterpret_cast<uint4*>(sub + sw128(tok, c16 + 1)) = make_uint4(cv[4], cv[5], cv[6], cv[7]);
  }
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_tc_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tile = smem;                 // Khat, f16, [128 tok] x [512 dims], 8 sub-tiles
  uint8_t* qop = smem + kTileBytes;     // Q, f16, [64 heads] x [512 dims], 8 sub-tiles
  uint8_t* pop = qop + kQBytes;         // P^T, f16, [128 tok] x [64 heads], MN-major
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kCtlOff);

  const int hg = blockIdx.y, r = blockIdx.z;
  const int split = blockIdx.x;
  const int nsplit = p.splits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = split * p.split_len;
  const int nj = max(0, min(p.split_len, p.topk - j0));
  const int ntiles = (nj + kTok - 1) / kTok;
  const bool report = hg == 0;
  const int head0 = hg * kHeads;
  const int nheads = min(kHeads, p.heads - head0);
  // Softmax role: lane quarter (tokens 32*quarter + lane of a tile) and the
  // 32 heads hh .. hh+31 this thread holds.
  const int quarter = warp & 3;
  const int hh = (warp >> 2) * 32;
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;

  grid_dep_launch();
  int len = p.rows.seq_lens[r];
  if (len < 0) {
    if (report && split == 0 && tid == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }

  // ---- set-up: barriers, TMEM
  if (tid == 0) {
    mbar_init(&ctl->bar_s, 1);
    mbar_init(&ctl->bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // ---- Q operand: 4 threads per head, 128 elements each; power-of-two scale
  // per head so every bf16 value is exact in f16.  Heads past the row's count
  // are zero.  (Q loads are issued first: they do not depend on the kernel
  // before.)
  const int qh = tid >> 2, qq = tid & 3;
  uint4 qraw[16];
  {
    const bool real = qh < nheads;
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (static_cast<int64_t>(r) * p.heads + head0 + qh) * 512 + qq * 128);
#pragma unroll
    for (int j = 0; j < 16; ++j) qraw[j] = real ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
  }
  grid_dep_wait();  // the selection comes from the kernel before

  // ---- slots of every entry of this split (two dependent loads each)
  {
    constexpr int kPer = kMaxTiles * kTok / kThreads;
    int idx[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      idx[i] = e < nj ? p.sel[static_cast<int64_t>(r) * p.topk + j0 + e] : -1;  // (after the wait)
    }
    const int32_t* bt = p.rows.block_table + static_cast<int64_t>(r) * p.rows.bt_stride;
    const int bs = p.rows.block_size;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      if (e >= kMaxTiles * kTok) break;
      int32_t slot = -1;
      const int t = idx[i];
      if (t != -1) {
        if (t < 0 || t >= len) {
          if (report) record_error(p.err, DSA_DEVERR_SELECT, r);
        } else {
          const int blk = t / bs;
          const int phys = blk < p.rows.max_blocks_per_seq ? __ldg(bt + blk) : -1;
          const int64_t s = static_cast<int64_t>(phys) * bs + t % bs;
          if (phys < 0 || s >= p.nslots) {
            if (report) record_error(p.err, DSA_DEVERR_BLOCK, r);
          } else {
            slot = static_cast<int32_t>(s);
          }
        }
      }
      ctl->slot[e] = slot;
    }
  }

  {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t w[4] = {qraw[j].x, qraw[j].y, qraw[j].z, qraw[j].w};
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
    if (qq == 0)
      ctl->qexp[qh] = p.sm_scale * p.kv_scale * 1.4426950408889634f * ldexpf(1.0f, -sh);
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // 8 elements = one 16-byte chunk of the operand
      const uint32_t w[4] = {qraw[j].x, qraw[j].y, qraw[j].z, qraw[j].w};
      uint32_t o4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o4[i] = pack_f16x2(__uint_as_float(w[i] << 16) * scale,
                           __uint_as_float(w[i] & 0xFFFF0000u) * scale);
      const int d0 = qq * 128 + j * 8;  // first of the 8 dims
      *reinterpret_cast<uint4*>(qop + (d0 >> 6) * kSubQ + sw128(qh, (d0 & 63) >> 3)) =
          make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }
  __syncthreads();  // slots, qexp visible
  const uint32_t tmem = ctl->tmem_base;

  uint4 raw[16];
  gather_tile(raw, ctl->slot, p.pool, 0, nj, warp, lane);

  bool alive = true;
  float m_run = -INFINITY;  // running max of head hh + lane (log2 units)
  float l_part = 0.0f;      // its sum over this lane quarter's tokens
  for (int it = 0; it < ntiles; ++it) {
    // ---- the tile buffer and P^T are free once the previous O^T MMAs are done
    if (it > 0) warp_wait(&ctl->bar_o, (it - 1) & 1, alive, lane, p.err, r);
    store_tile(tile, raw, warp, lane);
    if (it + 1 < ntiles) gather_tile(raw, ctl->slot, p.pool, (it + 1) * kTok, nj, warp, lane);
    fence_proxy_async_smem();  // generic-proxy operand writes -> visible to the tensor core
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- S^T = Khat Q^T (M = 128 tokens, N = 64 heads, K = 512)
    if (tid == 0) {
      const uint32_t idesc = idesc_f16(kTok, kHeads, false, false);
      const uint32_t a0 = smem_u32(tile), b0 = smem_u32(qop);
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const uint32_t a = a0 + (kk >> 2) * kSubTok + (kk & 3) * 32;
        const uint32_t b = b0 + (kk >> 2) * kSubQ + (kk & 3) * 32;
        umma_bf16(tmem, umma_desc_sw128_kmajor(a), umma_desc_sw128_kmajor(b), idesc, kk != 0);
      }
      umma_commit(&ctl->bar_s);
    }

    // ---- softmax of this tile
    warp_wait(&ctl->bar_s, it & 1, alive, lane, p.err, r);
    tc_fence_after();
    const int tok = quarter * 32 + lane;
    const int e = it * kTok + tok;
    const bool valid = e < nj && ctl->slot[e] >= 0;
    float z[32];
    tmem_load32(tmem + lane_base + hh, z);
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 qe = *reinterpret_cast<const float4*>(&ctl->qexp[hh + i]);
      z[i] = valid ? z[i] * qe.x : -INFINITY;
      z[i + 1] = valid ? z[i + 1] * qe.y : -INFINITY;
      z[i + 2] = valid ? z[i + 2] * qe.z : -INFINITY;
      z[i + 3] = valid ? z[i + 3] * qe.w : -INFINITY;
    }
    {
      float w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = z[i];
      ctl->red[quarter][hh + lane] = warp_transpose_reduce<true>(w, lane);
    }
    __syncthreads();
    const float tm = fmaxf(fmaxf(ctl->red[0][hh + lane], ctl->red[1][hh + lane]),
                           fmaxf(ctl->red[2][hh + lane], ctl->red[3][hh + lane]));
    float alpha = 1.0f;
    if (tm > m_run + kRescaleLog2) {  // also the first finite maximum (m_run = -inf)
      alpha = exp2f(m_run - tm);      // 0 while nothing was accumulated
      m_run = tm;
      l_part *= alpha;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float m = __shfl_sync(0xFFFFFFFFu, m_run, i);
      z[i] = z[i] == -INFINITY ? 0.0f : exp2f(z[i] - m);
    }
    {
      // P^T row `tok`: heads hh .. hh+31 = 16-byte chunks hh/8 .. hh/8+3.
      uint8_t* row = pop + tok * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(row + (((hh >> 3) + c) ^ (tok & 7)) * 16) =
            make_uint4(pack_f16x2(z[8 * c], z[8 * c + 1]), pack_f16x2(z[8 * c + 2], z[8 * c + 3]),
                       pack_f16x2(z[8 * c + 4], z[8 * c + 5]), pack_f16x2(z[8 * c + 6], z[8 * c + 7]));
    }
    l_part += warp_transpose_reduce<false>(z, lane);
    fence_proxy_async_smem();
    tc_fence_before();
    const int rescale = __syncthreads_or(it > 0 && alpha != 1.0f);
    tc_fence_after();
    if (rescale) {
      // O^T columns of the heads whose maximum moved, scaled in place.
      float a[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = __shfl_sync(0xFFFFFFFFu, alpha, i);
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        float v[32];
        const uint32_t taddr = tmem + lane_base + 64 + mb * 64 + hh;
        tmem_load32(taddr, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= a[i];
        tmem_store32(taddr, v);
      }
      tmem_store_wait();
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }

    // ---- O^T += V^T P^T (4 blocks of M = 128 dims, N = 64 heads, K = 128 tokens)
    if (tid == 0) {
      const uint32_t idesc = idesc_f16(128, kHeads, true, true);
      const uint32_t a0 = smem_u32(tile), b0 = smem_u32(pop);
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int kk = 0; kk < kTok / 16; ++kk) {
          // A: dims 128mb.. (two 64-dim sub-tiles, kSubTok apart), tokens 16kk..
          // B: tokens 16kk.. of P^T (one 64-head chunk per 128-byte row).
          const uint32_t a = a0 + (2 * mb) * kSubTok + kk * 2048;
          const uint32_t b = b0 + kk * 2048;
          umma_bf16(tmem + 64 + mb * 64, umma_desc_sw128_mnmajor(a, kSubTok),
                    umma_desc_sw128_mnmajor(b, kPBytes), idesc, (it > 0 || kk != 0) ? 1u : 0u);
        }
      }
      umma_commit(&ctl->bar_o);
    }
  }
  if (ntiles > 0) warp_wait(&ctl->bar_o, (ntiles - 1) & 1, alive, lane, p.err, r);
  tc_fence_after();

  // ---- per-head sums over the four lane quarters, in fixed order
  ctl->red[quarter][hh + lane] = l_part;
  __syncthreads();
  if (quarter == 0) {
    const int h = hh + lane;
    const float l = ((ctl->red[0][h] + ctl->red[1][h]) + ctl->red[2][h]) + ctl->red[3][h];
    ctl->lfin[h] = l;
    ctl->mfin[h] = m_run;
    if (nsplit > 1)
      reinterpret_cast<float2*>(p.part_ml)[((static_cast<int64_t>(r) * gridDim.y + hg) * nsplit +
                                            split) * kHeads + h] = make_float2(m_run, l);
    else if (p.lse != nullptr && h < nheads)
      p.lse[static_cast<int64_t>(r) * p.heads + head0 + h] =
          m_run != -INFINITY ? (m_run + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }

  // ---- O^T from TMEM, staged as rows [64 heads][512 dims] in the tile region
  {
    // Warp w reads lane quarter w%4 (dims 32*(w%4) + lane of each block) of
    // blocks mb = 2*(w/4), 2*(w/4)+1, all 64 heads (consecutive lanes ->
    // consecutive floats).
    float* stage = reinterpret_cast<float*>(tile);
    const int dl = quarter * 32 + lane;
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      const int mb = (warp >> 2) * 2 + bb;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[32];
        tmem_load32(tmem + lane_base + 64 + mb * 64 + hc * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i)  // (no tile ran: nothing was accumulated)
          stage[(hc * 32 + i) * 512 + mb * 128 + dl] = ntiles > 0 ? v[i] : 0.0f;
      }
    }
    tc_fence_before();
    __syncthreads();
    const float4* src = reinterpret_cast<const float4*>(stage);
    if (nsplit > 1) {
      // This split's partial rows, 16-byte coalesced stores (512 B per thread).
      float4* dst = reinterpret_cast<float4*>(
          p.part_o + ((static_cast<int64_t>(r) * gridDim.y + hg) * nsplit + split) * (kHeads * 512));
#pragma unroll 8
      for (int i = tid; i < kHeads * 128; i += kThreads) dst[i] = src[i];
    } else {
      // The only split: normalise, round to bf16, write the output rows.
#pragma unroll 4
      for (int i = tid; i < nheads * 128; i += kThreads) {
        const int h = i >> 7;
        const float l = ctl->lfin[h];
        const float scale = ctl->mfin[h] != -INFINITY ? p.kv_scale / l : 0.0f;
        const float4 v = src[i];
        uint2 packed;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed.x) : "f"(v.y * scale), "f"(v.x * scale));
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed.y) : "f"(v.w * scale), "f"(v.z * scale));
        reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(r) * p.heads + head0 + h) * 512)[i & 127] =
            packed;
      }
    }
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
  for (int c = 0; c < nsplit; ++c) mmax = fmaxf(mmax, ld_dep_f2(ml + (base + c) * kHeads + hl).x);
  float lsum = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (mmax != -INFINITY) {
    int c = 0;
    for (; c + 8 <= nsplit; c += 8) {  // eight splits' loads in flight at a time
      float2 mlc[8];
      float4 vc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        mlc[u] = ld_dep_f2(ml + (base + c + u) * kHeads + hl);
        vc[u] = ld_dep_f4(reinterpret_cast<const float4*>(p.part_o + ((base + c + u) * kHeads + hl) * 512) + tid);
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
      const float2 mlc = ld_dep_f2(ml + (base + c) * kHeads + hl);
      const float4 v = ld_dep_f4(reinterpret_cast<const float4*>(p.part_o + ((base + c) * kHeads + hl) * 512) + tid);
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
  const int target = (p.heads > kHeads ? 4 : 2) * kTok;
  int n = (p.topk + target - 1) / target;
  if (n < 1) n = 1;
  p.splits = n;
  p.split_len = (p.topk + n - 1) / n;
}

static int decode_splits(int32_t heads, int32_t topk) {
  DecodeParams p = {};
  p.heads = heads;
  p.topk = topk;
  plan_mla_decode_tc(p);
  return p.splits;
}

size_t mla_decode_tc_workspace_bytes(int32_t rows, int32_t heads, int32_t topk) {
  const int n = decode_splits(heads, topk);
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
  if (p.split_len > kMaxTiles * kTok) return cudaErrorInvalidValue;
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
  if (e != cudaSuccess || p.splits == 1) return e;
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
