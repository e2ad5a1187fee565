// mla_decode_tc.cu -- S3 on the 5th-generation tensor cores: absorbed NoPE
// MLA gather-attend with FP8 (kind::f8f6f4) tcgen05 MMAs, TMA row gathers and
// accumulators in TMEM.
//
// "glm5next_dsa/layer.rs": module header trap 4 (Q arrives absorbed into the
// 512-wide latent space), attend_rows (one launch for all rows, each with its
// own selection row, seq_len and block-table row; K and V are the same latent
// pool), decode_k (slot = block * block_size + pos % block_size).  Per row and
// head:  z_j = sm_scale * kv_scale * (Q . e4m3(latent_j)),  p = softmax(z),
//        out = kv_scale * sum_j p_j e4m3(latent_j),  lse = log sum_j exp(z_j).
//
// A row's selection is cut into n splits of at most 256 entries (512 when
// the caller asks for long splits, 2048 with more than 64 heads); n depends
// on topk, heads and that choice only, never on the number of rows, so a
// row's arithmetic is the same in any launch.  One CTA (20
// warps) runs one split of one (row, 64-head group) as a pipeline over
// 128-entry tiles:
//   - the latent stays FP8: TMA tile::gather4 copies the selected 512-byte
//     rows (4 rows x one 128-byte column block per copy, rows that are not
//     there zero-filled) straight into a 128-byte-swizzled tile, two tiles in
//     flight.  A warp issues these copies one after another, ~100 cycles
//     each, so three producer warps share the 128 copies of a tile (measured
//     with one tile in flight: one issuing warp reaches ~10 GB/s per SM, two
//     ~18, four ~30, where latency rather than issue is the limit);
//   - Q is held as two E4M3 terms per element, hi = e4m3(q*2^s) and
//     lo = e4m3(q*2^s - hi), which represent a bf16 q exactly (bf16 has 8
//     significant bits, each term 4, and the residual is a multiple of q's
//     last bit); the two terms are the N = 128 rows of one operand, so
//     S^T = Khat [Qhi|Qlo]^T is one M = 128 (tokens) x N = 128 x K = 512 MMA
//     chain whose two column halves add up to the exact logits (warp 3);
//   - S is double-buffered in TMEM, so the MMAs of tile t+1 run while sixteen
//     softmax warps (one token x 16 heads per thread) work on tile t.  The
//     softmax is bound by the latency of its dependent steps, not by the
//     exponential and conversion units: sixteen warps of 16 heads (four per
//     scheduler) run a tile in about two thirds of the time eight warps of
//     32 heads take, at 96 registers per thread;
//   - softmax: the running maximum m of a head only moves when a logit would
//     push p = 2^(z-m) past 2^8.75 (below the E4M3 maximum 448); it is then
//     set 8 below the new tile maximum (the O columns and sums of that head
//     are rescaled in TMEM).  p enters the O MMAs as two E4M3 terms (about
//     the precision of a bf16 p: relative error <= 2^-8, and values below
//     2^-10, i.e. 18 octaves under the head's maximum, drop out); the row
//     sums add the unrounded p;
//   - O^T += V^T P^T: V^T is the same FP8 tile read as an MN-major operand,
//     P^T the two 64-byte halves (hi, lo) of each 128-byte token row, two
//     accumulating MMA chains into the same TMEM columns.
// With one split the CTA normalises and writes the bf16 output (and lse)
// itself; otherwise the split's unnormalised O rows and its (max, sum) go to
// the workspace (L2-resident) and a merge kernel, chained by programmatic
// dependent launch, combines the n splits of every (row, head) in fixed split
// order and discards the L2 lines it consumed.
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 640;          // warps 0-2 gather, warp 3 MMA, warps 4-19 softmax
constexpr int kProducerWarps = 3;      // (20 warps keep 96 registers per thread)
constexpr int kMmaWarp = 3;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kSoftmaxThreads = 512;
constexpr int kHeads = 64;             // heads per CTA
constexpr int kHpt = 16;               // heads per softmax thread (one token each)
constexpr int kTok = 128;              // entries per tile (MMA M of S^T)
constexpr int kTilesPerSplit = 2;      // split length target (tiles), up to 64 heads
constexpr int kTilesPerSplitLong = 4;  // the same with the caller's long-splits flag
constexpr int kTilesPerSplitWide = 16; // the same with more than 64 heads (two head-group CTAs)
constexpr int kMaxTiles = 16;          // tiles per split the CTA can hold slots for
constexpr int kMergeHeads = 4;         // merge kernel: heads per CTA for many rows (64 threads a head)
constexpr int kMergeThreads = 64 * kMergeHeads;
constexpr float kPMaxLog2 = 8.75f;     // p = 2^(z - m) stays below 2^8.75 < 448
constexpr float kPResetLog2 = 8.0f;    // a reset maps the tile maximum to p = 2^8
constexpr uint32_t kSub = kTok * 128;              // one 128-dim column block: 128 rows x 128 B
constexpr uint32_t kTileBytes = 4 * kSub;          // FP8 latent tile: 64 KB
constexpr uint32_t kQBytes = 4 * kSub;             // Q operand: 128 rows (hi | lo) x 512 B
constexpr uint32_t kPBytes = kTok * 128;           // P^T: 128 token rows x (64 hi + 64 lo) B
constexpr uint32_t kTmemCols = 512;                // S buffers: cols 0..255, O^T: 256 + 64*mb
constexpr uint32_t kOCol = 256;

struct __align__(16) Ctl {
  uint64_t full[2], empty[2], sfull[2], sfree[2];
  uint64_t pready, odone, drain;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float qexp[kHeads];    // per-head logit scale (log2 units)
  alignas(16) float red[4][kHeads];  // per lane quarter: head maxima, then sums
  alignas(16) float mrun[kHeads];    // running maximum of each head (log2 units)
  int32_t slot[kMaxTiles * kTok];    // -1: no latent row (zero-filled by the gather)
};
constexpr uint32_t kCtlOff = 2 * kTileBytes + kQBytes + kPBytes;
constexpr uint32_t kSmemBytes = kCtlOff + sizeof(Ctl) + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Two floats to two E4M3 codes (round to nearest even, saturating): `lo` in
// the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(hi), "f"(lo));
  return out;
}
// The two codes decoded back to float (exact: E4M3 values are f16 values).
__device__ __forceinline__ float2 e4m3x2_decode(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}
// Descriptor of an MN-major operand in the 128-byte swizzled layout: 128
// contiguous bytes of MN per K row, K rows 128 B apart, the next 8 K rows
// 1024 bytes on, the next 128 bytes of MN `lbo` bytes on.
__device__ __forceinline__ uint64_t umma_desc_sw128_mnmajor(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// Instruction descriptor, kind::f8f6f4 with E4M3 A and B (format code 0),
// F32 accumulate; A and B each K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (a_mn_major ? (1u << 15) : 0u) | (b_mn_major ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem]^T on E4M3 operands, issued by one thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Four 128-byte rows (rows y0..y3, bytes x..x+127 of each) gathered by TMA
// into 512 consecutive bytes of shared memory (swizzled by address); rows
// outside the tensor are zero-filled.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y0, int32_t y1, int32_t y2,
                                            int32_t y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
      "r"(smem_u32(bar))
      : "memory");
}
// Drop a 128-byte L2 line without writing it back (its contents become
// undefined); used on partials that have been consumed.
__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}
// 16 consecutive TMEM columns of this thread's lane (waited in the same asm).
__device__ __forceinline__ void tmem_load16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_store16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Named barrier of the 256 softmax threads (id 1); the second form returns
// whether any of them passed a true predicate.
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
}
__device__ __forceinline__ bool softmax_sync_or(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "n"(kSoftmaxThreads)
      : "memory");
  return out != 0;
}

// One butterfly step of a warp transpose-reduction: on entry v[0..2S) are
// values of 2S heads in this lane; on exit v[0..S) hold, for the S heads
// selected by lane bit S, the reduction over this lane and lane ^ S.
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
// The steps S = 8, 4, 2, 1 on 16 heads, then lanes l and l ^ 16 combined:
// v[0] of lane l ends as the reduction of head l % 16 over the 32 lanes, in an
// order fixed by the lane numbering (lanes l and l ^ 16 hold the same value).
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce16(float (&v)[16], int lane) {
  butterfly_step<8, kMax>(v, lane);
  butterfly_step<4, kMax>(v, lane);
  butterfly_step<2, kMax>(v, lane);
  butterfly_step<1, kMax>(v, lane);
  const float o = __shfl_xor_sync(0xFFFFFFFFu, v[0], 16);
  return kMax ? fmaxf(v[0], o) : v[0] + o;
}

__device__ __forceinline__ void set_abort(Ctl* c) {
  *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}
__device__ __forceinline__ bool aborted(Ctl* c) {
  return *reinterpret_cast<volatile int*>(&c->abort_flag) != 0;
}
// Bounded wait of a whole warp on an mbarrier phase (lane 0 polls).  A
// timeout is recorded, the CTA is marked aborted and false is returned.
__device__ __forceinline__ bool warp_wait(Ctl* c, uint64_t* bar, uint32_t parity, int lane,
                                          int* err, int r, uint64_t limit_ns) {
  int ok = 1;
  if (lane == 0) {
    ok = aborted(c) ? 0 : (mbar_wait(bar, parity, limit_ns) ? 1 : 0);
    if (!ok && !aborted(c)) {
      record_error(err, DSA_DEVERR_TIMEOUT, r);
      set_abort(c);
    }
  }
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap pmap, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = smem;                       // 2 x FP8 latent tile [128 tok][512 B]
  uint8_t* qop = smem + 2 * kTileBytes;        // [Qhi 64 rows | Qlo 64 rows] x 512 B
  uint8_t* pop = qop + kQBytes;                // P^T: [128 tok][64 hi | 64 lo] B
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

  grid_dep_launch();

  // ---- set-up: barriers, TMEM (nothing here reads an input)
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
      mbar_init(&ctl->sfull[s], 1);
      mbar_init(&ctl->sfree[s], kSoftmaxThreads / 32);
    }
    mbar_init(&ctl->pready, kSoftmaxThreads / 32);
    mbar_init(&ctl->odone, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&pmap);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid < kHeads) ctl->mrun[tid] = -INFINITY;
  // Q may be the output of the kernel before (a projection), so by default it
  // is only prefetched into L2 here (a prefetch cannot make a later load
  // stale) and loaded after the dependency wait.  With q_early the caller has
  // declared Q complete before the kernel before this one started, and Q is
  // loaded and converted now, while that kernel runs.  Warp w converts heads
  // w, w+20, ...; lane l dims 16l..16l+15 (32 bytes: lanes 4i..4i+3 share a
  // 128-byte line).
  constexpr int kQPer = (kHeads + kThreads / 32 - 1) / (kThreads / 32);
  uint4 qa[kQPer], qb[kQPer];
  auto load_q = [&]() {
#pragma unroll
    for (int j = 0; j < kQPer; ++j) {
      const int h = warp + j * (kThreads / 32);
      if (h < nheads) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (static_cast<int64_t>(r) * p.heads + head0 + h) * 512 + lane * 16);
        qa[j] = ld_dep_u4(src);
        qb[j] = ld_dep_u4(src + 1);
      } else {
        qa[j] = make_uint4(0, 0, 0, 0);
        qb[j] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // ---- Q operand: q*2^s = hi + lo (E4M3 each), s a power of two per head
  // putting the head's largest |q| in [128, 256).  Row h holds hi, row 64+h lo.
  auto convert_q = [&]() {
#pragma unroll
    for (int j = 0; j < kQPer; ++j) {
      const int h = warp + j * (kThreads / 32);
      if (h >= kHeads) break;
      const uint32_t w[8] = {qa[j].x, qa[j].y, qa[j].z, qa[j].w, qb[j].x, qb[j].y, qb[j].z, qb[j].w};
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      int e = 0;
      if (amax > 0.0f) frexpf(amax, &e);  // amax < 2^e
      const int sh = max(-100, min(100, 8 - e));
      const float scale = ldexpf(1.0f, sh);
      if (lane == 0)
        ctl->qexp[h] = p.sm_scale * p.kv_scale * 1.4426950408889634f * ldexpf(1.0f, -sh);
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint16_t hc[2], lc[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float a0 = x[4 * i + 2 * k] * scale, a1 = x[4 * i + 2 * k + 1] * scale;
          hc[k] = e4m3x2(a0, a1);
          const float2 hv = e4m3x2_decode(hc[k]);
          lc[k] = e4m3x2(a0 - hv.x, a1 - hv.y);
        }
        hw[i] = static_cast<uint32_t>(hc[0]) | (static_cast<uint32_t>(hc[1]) << 16);
        lw[i] = static_cast<uint32_t>(lc[0]) | (static_cast<uint32_t>(lc[1]) << 16);
      }
      // Dims 16l..16l+15 = 16-byte chunk l%8 of column block l/8.
      uint8_t* blk = qop + (lane >> 3) * kSub;
      const uint32_t c = static_cast<uint32_t>(((lane & 7) ^ (h & 7)) * 16);
      *reinterpret_cast<uint4*>(blk + h * 128 + c) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(blk + (h + kHeads) * 128 + c) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  };
  const bool q_early =
      static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(gridDim.x) * (blockIdx.y + static_cast<int64_t>(gridDim.y) * blockIdx.z) <
      p.q_early;
  if (q_early) {
    load_q();
    convert_q();
  } else {
#pragma unroll
    for (int j = 0; j < kQPer; ++j) {
      const int h = warp + j * (kThreads / 32);
      if (h < nheads && (lane & 3) == 0)
        prefetch_l2(p.q + (static_cast<int64_t>(r) * p.heads + head0 + h) * 512 + lane * 16);
    }
  }
  grid_dep_wait();  // the selection (and possibly Q, seq_lens) come from kernels before

  int len = p.rows.seq_lens[r];
  if (len < 0) {
    if (report && split == 0 && tid == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }
  if (!q_early) load_q();
  // The split's selection entries, issued before the Q conversion so both
  // round trips overlap.
  constexpr int kPer = (kMaxTiles * kTok + kThreads - 1) / kThreads;
  int idx[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = tid + i * kThreads;
    idx[i] = e < nj ? p.sel[static_cast<int64_t>(r) * p.topk + j0 + e] : -1;  // plain load
  }
  if (!q_early) convert_q();

  // ---- slots of every entry of this split (a table lookup each)
  {
    const int32_t* bt = p.rows.block_table + static_cast<int64_t>(r) * p.rows.bt_stride;
    const int bs = p.rows.block_size;
    // All table lookups in flight before any is used (one round trip).
    int phys[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int t = idx[i];
      const int blk = t >= 0 && t < len ? t / bs : -1;
      phys[i] = (blk >= 0 && blk < p.rows.max_blocks_per_seq) ? bt[blk] : -1;  // plain load
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = tid + i * kThreads;
      if (e >= ntiles * kTok) break;  // the tiles of this split only
      int32_t slot = -1;
      const int t = idx[i];
      if (t != -1) {
        if (t < 0 || t >= len) {
          if (report) record_error(p.err, DSA_DEVERR_SELECT, r);
        } else {
          const int64_t s = static_cast<int64_t>(phys[i]) * bs + t % bs;
          if (phys[i] < 0 || s >= p.nslots) {
            if (report) record_error(p.err, DSA_DEVERR_BLOCK, r);
          } else {
            slot = static_cast<int32_t>(s);
          }
        }
      }
      ctl->slot[e] = slot;
    }
  }

  fence_proxy_async_smem();  // generic-proxy operand writes -> visible to the tensor core
  tc_fence_before();
  __syncthreads();           // slots, qexp, Q operand, barriers, TMEM address
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // ---- the first two tiles (both ring stages are free) are gathered by every
  // warp but the MMA warp: the softmax warps have nothing to do before the
  // first S is ready, and each warp issues its copies one after another.
  // Copy g of the pair is issued by warp g % 19, lane g / 19 (tile 0's copies
  // come first in every warp).
  const int first = min(ntiles, 2);
  if (warp != kMmaWarp) {
    constexpr int kIssuerWarps = kThreads / 32 - 1;
    const int widx = warp < kMmaWarp ? warp : warp - 1;
    if (widx == 0 && lane == 0)
      for (int t = 0; t < first; ++t) mbar_arrive_expect_tx(&ctl->full[t], kTileBytes);
    for (int g = widx + kIssuerWarps * lane; g < first * 128; g += kIssuerWarps * 32) {
      const int t = g >> 7, gg = g & 127;
      const int rg = gg >> 2, sb = gg & 3;
      const int32_t* sl = ctl->slot + t * kTok + 4 * rg;
      tma_gather4(smem_u32(tiles + t * kTileBytes + sb * kSub + rg * 512), &pmap, &ctl->full[t],
                  sb * 128, sl[0], sl[1], sl[2], sl[3]);
    }
  }

  if (warp < kProducerWarps) {
    // ================================================================ gather
    // Tiles from the third on.  Copy g (0..127) of a tile moves rows
    // 4(g/4) .. 4(g/4)+3 of the tile, column block g%4; producer warp w
    // issues copies w, w+3, w+6, ... (43, 43 and 42 of them), lane l the ones
    // with index w + 3(l + 32j).  Warp 0 lane 0 posts the tile's byte count;
    // other copies may land before it does (the transaction count may run
    // ahead of the expectation).
    int issued = first;
    for (int t = first; t < ntiles; ++t) {
      const int s = t & 1;
      if (!warp_wait(ctl, &ctl->empty[s], ((t - 2) >> 1) & 1, lane, p.err, r, p.wait_ns)) break;
      if (warp == 0 && lane == 0) mbar_arrive_expect_tx(&ctl->full[s], kTileBytes);
      for (int g = warp + kProducerWarps * lane; g < 128; g += kProducerWarps * 32) {
        const int rg = g >> 2, sb = g & 3;
        const int32_t* sl = ctl->slot + t * kTok + 4 * rg;
        tma_gather4(smem_u32(tiles + s * kTileBytes + sb * kSub + rg * 512), &pmap, &ctl->full[s],
                    sb * 128, sl[0], sl[1], sl[2], sl[3]);
      }
      issued = t + 1;
    }
    // Never leave with a copy in flight: wait (bounded) for the last gathers
    // (already complete unless the pipeline gave up).
    if (warp == 0 && lane == 0)
      for (int t = max(0, issued - 2); t < issued; ++t)
        mbar_wait(&ctl->full[t & 1], (t >> 1) & 1, kDrainWaitNs);
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_e4m3(kTok, 2 * kHeads, false, false);
      const uint32_t idesc_o = idesc_e4m3(128, kHeads, true, true);
      const uint32_t q0 = smem_u32(qop), p0 = smem_u32(pop);
      auto issue_o = [&](int u) {
        const uint32_t a0 = smem_u32(tiles + (u & 1) * kTileBytes);
#pragma unroll
        for (int term = 0; term < 2; ++term)
#pragma unroll
          for (int mb = 0; mb < 4; ++mb)
#pragma unroll
            for (int kk = 0; kk < kTok / 32; ++kk) {
              // A: dims 128mb.. (one 128-byte column block), tokens 32kk..
              // B: tokens 32kk.. of P^T, heads as the hi or lo 64 bytes.
              const uint32_t a = a0 + mb * kSub + kk * 4096;
              const uint32_t b = p0 + kk * 4096 + term * 64;
              umma_e4m3(tmem + kOCol + mb * kHeads, umma_desc_sw128_mnmajor(a, kSub),
                        umma_desc_sw128_mnmajor(b, kPBytes), idesc_o,
                        (u > 0 || term > 0 || kk > 0) ? 1u : 0u);
            }
      };
      // Event-driven issue: O(u) goes out as soon as the softmax of tile u is
      // done (it frees a ring stage for the gather), S(t) as soon as tile t has
      // landed and its S buffer is free; neither waits behind the other.
      int ns = 0, no = 0;  // next S and next O to issue
      uint64_t t_last = global_ns();
      uint32_t idle = 0;
      while (no < ntiles) {
        bool issued = false;
        if (no < ns && mbar_try_wait(&ctl->pready, no & 1)) {
          tc_fence_after();
          issue_o(no);
          umma_commit(&ctl->empty[no & 1]);
          umma_commit(&ctl->odone);
          ++no;
          issued = true;
        } else if (ns < ntiles && mbar_try_wait(&ctl->full[ns & 1], (ns >> 1) & 1) &&
                   (ns < 2 || mbar_try_wait(&ctl->sfree[ns & 1], ((ns - 2) >> 1) & 1))) {
          tc_fence_after();
          // S^T (cols 128s..): M = 128 tokens, N = 128 (64 heads hi | 64 lo), K = 512
          const int s = ns & 1;
          const uint32_t a0 = smem_u32(tiles + s * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint32_t a = a0 + (kk >> 2) * kSub + (kk & 3) * 32;
            const uint32_t b = q0 + (kk >> 2) * kSub + (kk & 3) * 32;
            umma_e4m3(tmem + s * 2 * kHeads, umma_desc_sw128_kmajor(a), umma_desc_sw128_kmajor(b),
                      idesc_s, kk != 0);
          }
          umma_commit(&ctl->sfull[s]);
          ++ns;
          issued = true;
        }
        if (issued) {
          idle = 0;
          t_last = global_ns();
        } else if ((++idle & 255u) == 0) {
          if (aborted(ctl)) break;
          if (global_ns() - t_last > p.wait_ns) {
            record_error(p.err, DSA_DEVERR_TIMEOUT, r);
            set_abort(ctl);
            break;
          }
        }
      }
      // Every MMA issued by this thread is complete before TMEM is released.
      umma_commit(&ctl->drain);
      mbar_wait(&ctl->drain, 0, kDrainWaitNs);
    }
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0) {
    // ================================================================ softmax
    // Every softmax warp passes the same named barriers in the same order
    // whatever happens (a timed-out wait only makes the warp skip work), so a
    // timeout can never leave a barrier short of threads.  Softmax warp w
    // (0..15) reads TMEM lanes 32*(w%4).. (its tokens) and heads 16*(w/4)..;
    // lane l reduces for head hh + l%16.
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. = tokens
    const int hh = ((warp - kSoftmaxWarp0) >> 2) * kHpt;  // heads hh .. hh+15
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int tok = quarter * 32 + lane;
    const int hl = hh + (lane & (kHpt - 1));
    float ls[kHpt];                               // this token lane's share of each head's sum
#pragma unroll
    for (int i = 0; i < kHpt; ++i) ls[i] = 0.0f;
    float m_lane = -INFINITY;  // running maximum of head hl (log2 units)
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int b = t & 1;
      float z[kHpt];
      if (ok) ok = warp_wait(ctl, &ctl->sfull[b], (t >> 1) & 1, lane, p.err, r, p.wait_ns);
      if (ok) {
        float zl[kHpt];
        tc_fence_after();
        tmem_load16(tmem + lane_base + b * 2 * kHeads + hh, z);
        tmem_load16(tmem + lane_base + b * 2 * kHeads + kHeads + hh, zl);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->sfree[b]);
        const int e = t * kTok + tok;
        const bool valid = e < nj && ctl->slot[e] >= 0;
#pragma unroll
        for (int i = 0; i < kHpt; i += 4) {
          const float4 qe = *reinterpret_cast<const float4*>(&ctl->qexp[hh + i]);
          z[i] = valid ? (z[i] + zl[i]) * qe.x : -INFINITY;
          z[i + 1] = valid ? (z[i + 1] + zl[i + 1]) * qe.y : -INFINITY;
          z[i + 2] = valid ? (z[i + 2] + zl[i + 2]) * qe.z : -INFINITY;
          z[i + 3] = valid ? (z[i + 3] + zl[i + 3]) * qe.w : -INFINITY;
        }
      } else {
#pragma unroll
        for (int i = 0; i < kHpt; ++i) z[i] = -INFINITY;
      }
      bool exceed = false;
#pragma unroll
      for (int i = 0; i < kHpt; i += 4) {
        const float4 mr = *reinterpret_cast<const float4*>(&ctl->mrun[hh + i]);
        exceed |= z[i] > mr.x + kPMaxLog2;
        exceed |= z[i + 1] > mr.y + kPMaxLog2;
        exceed |= z[i + 2] > mr.z + kPMaxLog2;
        exceed |= z[i + 3] > mr.w + kPMaxLog2;
      }
      bool waited_o = false;
      if (softmax_sync_or(exceed)) {
        // Tile maximum of every head, then the new running maxima.
        {
          float w[kHpt];
#pragma unroll
          for (int i = 0; i < kHpt; ++i) w[i] = z[i];
          const float tq = warp_transpose_reduce16<true>(w, lane);
          if (lane < kHpt) ctl->red[quarter][hl] = tq;
        }
        softmax_sync();
        const float tm = fmaxf(fmaxf(ctl->red[0][hl], ctl->red[1][hl]),
                               fmaxf(ctl->red[2][hl], ctl->red[3][hl]));
        float alpha = 1.0f;
        if (tm > m_lane + kPMaxLog2) {
          const float mn = tm - kPResetLog2;
          alpha = exp2f(m_lane - mn);  // 0 while nothing was accumulated
          m_lane = mn;
        }
        float a[kHpt];
#pragma unroll
        for (int i = 0; i < kHpt; ++i) {
          a[i] = __shfl_sync(0xFFFFFFFFu, alpha, i);
          ls[i] *= a[i];
        }
        if (ok && t > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
          // O^T columns of the heads whose maximum moved, scaled in place once
          // the previous tile's O MMAs are complete.
          ok = warp_wait(ctl, &ctl->odone, (t - 1) & 1, lane, p.err, r, p.wait_ns);
          waited_o = true;
          if (ok) {
            tc_fence_after();
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
              float v[kHpt];
              const uint32_t taddr = tmem + lane_base + kOCol + mb * kHeads + hh;
              tmem_load16(taddr, v);
#pragma unroll
              for (int i = 0; i < kHpt; ++i) v[i] *= a[i];
              tmem_store16(taddr, v);
            }
            tmem_store_wait();
          }
        }
        softmax_sync();                        // every warp has read red[] and the old mrun
        if (quarter == 0 && lane < kHpt) ctl->mrun[hl] = m_lane;
        softmax_sync();                        // the new mrun is visible
      }
      // p = 2^(z - m) as two E4M3 terms (hi, lo); the sums add the unrounded p.
      uint32_t hiw[kHpt / 4], low[kHpt / 4];
#pragma unroll
      for (int i = 0; i < kHpt; i += 4) {
        const float4 mr = *reinterpret_cast<const float4*>(&ctl->mrun[hh + i]);
        const float mm[4] = {mr.x, mr.y, mr.z, mr.w};
        uint16_t hc[2], lc[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = i + 2 * k;
          const float p0 = z[j] == -INFINITY ? 0.0f : exp2f(z[j] - mm[2 * k]);
          const float p1 = z[j + 1] == -INFINITY ? 0.0f : exp2f(z[j + 1] - mm[2 * k + 1]);
          hc[k] = e4m3x2(p0, p1);
          const float2 hv = e4m3x2_decode(hc[k]);
          lc[k] = e4m3x2(p0 - hv.x, p1 - hv.y);
          ls[j] += p0;
          ls[j + 1] += p1;
        }
        hiw[i >> 2] = static_cast<uint32_t>(hc[0]) | (static_cast<uint32_t>(hc[1]) << 16);
        low[i >> 2] = static_cast<uint32_t>(lc[0]) | (static_cast<uint32_t>(lc[1]) << 16);
      }
      // The P buffer is free once the previous tile's O MMAs are complete.
      if (ok && t > 0 && !waited_o) ok = warp_wait(ctl, &ctl->odone, (t - 1) & 1, lane, p.err, r, p.wait_ns);
      if (ok) {
        // P^T row `tok`: hi bytes of heads hh.. = chunk hh/16; lo = chunk 4 + hh/16.
        uint8_t* row = pop + tok * 128;
        const int c0 = hh >> 4, sw = tok & 7;
        *reinterpret_cast<uint4*>(row + ((c0 ^ sw) * 16)) = make_uint4(hiw[0], hiw[1], hiw[2], hiw[3]);
        *reinterpret_cast<uint4*>(row + (((c0 + 4) ^ sw) * 16)) = make_uint4(low[0], low[1], low[2], low[3]);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->pready);
      }
    }

    // ---- epilogue: per-head sums in fixed order (while the last O MMAs
    // run), then the output once they are complete
    const float l_quarter = warp_transpose_reduce16<false>(ls, lane);
    if (lane < kHpt) ctl->red[quarter][hl] = l_quarter;
    softmax_sync();
    const float l_lane = ((ctl->red[0][hl] + ctl->red[1][hl]) + ctl->red[2][hl]) + ctl->red[3][hl];
    if (quarter == 0 && lane < kHpt) {
      if (nsplit > 1)
        reinterpret_cast<float2*>(p.part_ml)[((static_cast<int64_t>(r) * gridDim.y + hg) * nsplit +
                                              split) * kHeads + hl] = make_float2(m_lane, l_lane);
      else if (p.lse != nullptr && hl < nheads)
        p.lse[static_cast<int64_t>(r) * p.heads + head0 + hl] =
            m_lane != -INFINITY ? (m_lane + log2f(l_lane)) * 0.69314718055994531f : -INFINITY;
    }
    // O^T: lane = dim 128mb + 32*quarter + lane, column = head.  For a fixed
    // head the 32 lanes write 32 consecutive dims.  One split: the output,
    // kv_scale * O / l, in bf16.  Several: the split's O / l in fp16 -- a
    // convex combination of E4M3 latent values, so |O / l| <= 448 and fp16
    // keeps it to 2^-11 relative, at half the bytes of FP32 (the stores of
    // the partials bound this epilogue) -- with (max, sum) beside it.
    const float sc_lane =
        (m_lane != -INFINITY && l_lane > 0.0f) ? (nsplit > 1 ? 1.0f : p.kv_scale) / l_lane : 0.0f;
    float sc[kHpt];
#pragma unroll
    for (int i = 0; i < kHpt; ++i) sc[i] = __shfl_sync(0xFFFFFFFFu, sc_lane, i);
    if (ok && ntiles > 0) ok = warp_wait(ctl, &ctl->odone, (ntiles - 1) & 1, lane, p.err, r, p.wait_ns);
    tc_fence_after();
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      float v[kHpt];
      const int d = mb * 128 + quarter * 32 + lane;
      if (ok && ntiles > 0) {  // (ok is uniform over the warp: tcgen05.ld is warp-collective)
        tmem_load16(tmem + lane_base + kOCol + mb * kHeads + hh, v);
      } else {
#pragma unroll
        for (int i = 0; i < kHpt; ++i) v[i] = 0.0f;
      }
      if (nsplit > 1) {
        uint16_t* dst = p.part_o + ((static_cast<int64_t>(r) * gridDim.y + hg) * nsplit + split) *
                                       (kHeads * 512) + d;
#pragma unroll
        for (int i = 0; i < kHpt; ++i) dst[(hh + i) * 512] = __half_as_ushort(__float2half_rn(v[i] * sc[i]));
      } else {
        uint16_t* dst = p.out + (static_cast<int64_t>(r) * p.heads + head0) * 512 + d;
#pragma unroll
        for (int i = 0; i < kHpt; ++i)
          if (hh + i < nheads)
            dst[(hh + i) * 512] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i] * sc[i]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One split's share of a merged (row, head): weight w = l * 2^(m - mmax) on
// the split's O / l (eight fp16 values).
__device__ __forceinline__ void accumulate_split(float2 ml, uint4 v, float mmax, float& lsum,
                                                 float (&acc)[8]) {
  const float w = ml.y * exp2f(ml.x - mmax);
  const uint32_t h[4] = {v.x, v.y, v.z, v.w};
  lsum += w;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
    acc[2 * k] += a.x * w;
    acc[2 * k + 1] += a.y * w;
  }
}

// Merge of the n splits of (row, head): blockDim.x / 64 heads per CTA (one
// for a few rows, four for many), 64 threads a head and 8 dims a thread,
// splits in fixed order; the consumed partial lines are discarded from L2.
// The arithmetic of an element does not depend on the mapping.
__global__ void __launch_bounds__(kMergeThreads) mla_decode_merge_kernel(const DecodeParams p) {
  const int tid = threadIdx.x, d8 = tid % 64;
  const int h = blockIdx.x * (blockDim.x / 64) + tid / 64, r = blockIdx.y;
  const int groups = (p.heads + kHeads - 1) / kHeads;
  const int hg = h / kHeads, hl = h % kHeads;
  const int nsplit = p.splits;
  const int64_t base = (static_cast<int64_t>(r) * groups + hg) * nsplit;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
  // The successor (the next step's indexer) may start now: a kernel that
  // reads what this one writes waits for it in any case, and an indexer whose
  // caller declared its inputs ready scores its keys while the attend and
  // this merge finish.
  grid_dep_launch();
  grid_dep_wait();  // the partials come from the kernel before
  if (h >= p.heads) return;  // (heads is a multiple of 16: never)
  float mmax = -INFINITY;
  float lsum = 0.0f;
  float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  auto row_of = [&](int u) {
    return reinterpret_cast<const uint4*>(p.part_o + ((base + u) * kHeads + hl) * 512) + d8;
  };
  if (nsplit <= 8) {
    // Every split's (max, sum) and partial row in flight at once: one round trip.
    float2 mlc[8];
    uint4 vc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < nsplit) {
        mlc[u] = ld_dep_f2(ml + (base + u) * kHeads + hl);
        vc[u] = ld_dep_u4(row_of(u));
      } else {
        mlc[u] = make_float2(-INFINITY, 0.0f);
        vc[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) mmax = fmaxf(mmax, mlc[u].x);
    if (mmax != -INFINITY) {
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u < nsplit) accumulate_split(mlc[u], vc[u], mmax, lsum, acc);
    }
  } else {
    // Maxima first (eight loads in flight per round), then the rows.
    for (int c0 = 0; c0 < nsplit; c0 += 8) {
      float m8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        m8[u] = c0 + u < nsplit ? ld_dep_f2(ml + (base + c0 + u) * kHeads + hl).x : -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) mmax = fmaxf(mmax, m8[u]);
    }
    if (mmax != -INFINITY) {
      for (int c0 = 0; c0 < nsplit; c0 += 8) {
        float2 mlc[8];
        uint4 vc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (c0 + u < nsplit) {
            mlc[u] = ld_dep_f2(ml + (base + c0 + u) * kHeads + hl);
            vc[u] = ld_dep_u4(row_of(c0 + u));
          }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (c0 + u < nsplit) accumulate_split(mlc[u], vc[u], mmax, lsum, acc);
      }
    }
  }
  const float scale = (mmax != -INFINITY && lsum > 0.0f) ? p.kv_scale / lsum : 0.0f;
  uint32_t packed[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(packed[k])
        : "f"(acc[2 * k + 1] * scale), "f"(acc[2 * k] * scale));
  const int64_t head = static_cast<int64_t>(r) * p.heads + h;
  // Two 8-byte stores (out is only required to be 8-byte aligned).
  uint2* o2 = reinterpret_cast<uint2*>(p.out + head * 512 + d8 * 8);
  o2[0] = make_uint2(packed[0], packed[1]);
  o2[1] = make_uint2(packed[2], packed[3]);
  if (d8 == 0 && p.lse != nullptr)
    p.lse[head] = mmax != -INFINITY ? (mmax + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
  // Every lane has used its partial values: drop the consumed 128-byte lines
  // (eight lanes of one warp share one) from L2 instead of writing them back.
  __syncwarp();
  if ((d8 & 7) == 0)
    for (int c = 0; c < nsplit; ++c)
      discard_l2_line(p.part_o + ((base + c) * kHeads + hl) * 512 + d8 * 8);
}

}  // namespace

void plan_mla_decode_tc(DecodeParams& p) {
  // A function of topk, heads and the caller's long-splits choice only, so a
  // row's arithmetic does not depend on the other rows of the launch.
  const int target = (p.heads > kHeads ? kTilesPerSplitWide
                                       : (p.long_splits ? kTilesPerSplitLong : kTilesPerSplit)) * kTok;
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
  const size_t o_bytes = (units * 512 * sizeof(uint16_t) + 255) & ~static_cast<size_t>(255);
  return o_bytes + units * 2 * sizeof(float);
}

void mla_decode_tc_bind_workspace(DecodeParams& p, void* workspace) {
  const size_t units =
      static_cast<size_t>(p.rows.rows) * ((p.heads + kHeads - 1) / kHeads) * p.splits * kHeads;
  p.part_o = static_cast<uint16_t*>(workspace);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       ((units * 512 * sizeof(uint16_t) + 255) & ~static_cast<size_t>(255)));
}

cudaError_t launch_mla_decode_tc(const DecodeParams& p, const CUtensorMap& pmap,
                                 cudaStream_t stream) {
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
  e = cudaLaunchKernelEx(&cfg, mla_decode_tc_kernel, pmap, p);
  if (e != cudaSuccess || p.splits == 1) return e;
  cudaLaunchConfig_t mcfg = {};
  // One head per CTA while that gives fewer than four CTAs per SM (a single
  // row: the most SMs), four per CTA beyond.
  const int hpc = static_cast<int64_t>(p.rows.rows) * p.heads >= 4LL * p.num_sms ? kMergeHeads : 1;
  mcfg.gridDim = dim3((p.heads + hpc - 1) / hpc, p.rows.rows, 1);
  mcfg.blockDim = dim3(64 * hpc, 1, 1);
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
// attend: a decode loop that must not pay cudaMalloc's implicit device
// synchronisation, and code whose device memory belongs to an allocator it may
// not call.  This entry point runs the same kernel as dsa_mla_decode_fp8 with
// the split partials in this file-scope device array instead of a
// caller-provided workspace.  The array is DSA_NOALLOC_SCRATCH_BYTES long and
// every GPU that loads the library keeps it until the process exits.  Every
// call shares it: calls that overlap on the GPU race on it.
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
