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
// Work split.  The rows of a sequence form launch groups of at most 64 score
// columns; group g has T_g = ceil(max row length / 128) key tiles.  The
// launch is persistent: about two CTAs per SM, and CTA c scores the tiles
// [c*T/C, (c+1)*T/C) of the concatenation of every group's tiles (T tiles in
// all), so every CTA gets the same number of tiles however the lengths are
// spread, and streams its keys from one set-up.  After the dependency wait
// every CTA sums T_g over the groups (the row lengths are device data) and
// finds where its range starts; its range then runs through one group or a
// few consecutive ones ("segments"), and the q operand is rebuilt at each
// segment boundary.  CTAs that score the same tiles for different groups of
// one sequence run concurrently and share the key tiles through L2.
//
// CTA roles (192 threads):
//   warp 0     walks the CTA's segments (row lengths checked per segment,
//              one record per segment in a small ring) and issues the key
//              TMA loads (lane 0);
//   warp 1     owns TMEM and issues the MMAs (lane 0);
//   warps 2-5  build each segment's q operand and head weights, then run the
//              epilogue (one TMEM lane quarter each).
// The arithmetic of every score is the same whichever CTA or segment
// computes it, so a row's scores do not depend on the other rows.
#include <climits>

#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kTileM = 128;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;  // warps 2-5
constexpr int kMaxStages = 6;
constexpr int kMaxSubRows = 32;
constexpr int kSegRing = 4;       // segment records in flight
constexpr int kDirectTiles = 2;   // tiles per CTA of a direct launch
constexpr int kScanThreads = 64;  // warps 0-1 find the CTA's range
constexpr int kScanRegs = 8;      // groups per scan thread kept between the two passes

struct Seg {
  int64_t base;        // arena row of the sequence's token 0
  int r0, nrows;       // the group's rows
  int t_first;         // first tile of the segment, counted within the group
  int ntiles;          // tiles in the segment
  int max_len;         // longest row of the group (tokens past it are not scored)
  int row_len[kMaxSubRows];
};

struct __align__(8) IndexCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qready;
  uint64_t segfull[kSegRing];
  uint64_t segfree[kSegRing];
  uint64_t drain;
  long long scan[kScanThreads / 32];
  long long my_tiles;
  uint32_t tmem_base;
  int abort_flag;
  int g0, t0;          // the group holding this CTA's first tile, and the tile within it
  int tg0;             // that group's tile count
  int64_t base0;       // and its arena base
  Seg seg[kSegRing];
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

// Named barrier of the four epilogue warps, returning the OR of `pred` over
// them (the same value in every thread, so they all leave a loop together).
__device__ __forceinline__ bool epi_sync_or(bool pred) {
  int out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1 : 0), "n"(kEpiThreads)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane, one wait for all.
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

// ---------------------------------------------------------------- launch groups
struct GroupRows {
  int seq, seq_row0, r0, nrows;
};
__device__ __forceinline__ GroupRows group_rows(const IndexParams& p, int g) {
  GroupRows gr;
  gr.seq = g / p.subs_per_seq;
  const int sub = g - gr.seq * p.subs_per_seq;
  gr.seq_row0 = gr.seq * p.rows_per_seq;
  gr.r0 = gr.seq_row0 + sub * p.sub_rows;
  gr.nrows = min(p.sub_rows, gr.seq_row0 + p.rows_per_seq - gr.r0);
  return gr;
}

// A row's scored length: its sequence length if the row is well formed, else
// 0 (and the reason recorded when `report`).  Every key row of a sequence
// lives at idx_base[first row of the sequence] + token.
__device__ __forceinline__ int row_len_checked(const IndexParams& p, int r, int64_t base,
                                               int written, bool report) {
  const int len = p.seq_lens[r];
  const int64_t rb = p.idx_base[r];
  if (len < 0 || len > p.max_len) {
    if (report) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    return 0;
  }
  if (rb != base || base < 0 || base + len > p.idx_tokens) {
    if (report) record_error(p.err, DSA_DEVERR_ARENA, r);
    return 0;
  }
  if (len > written) {  // the sequence's keys stop before this row's range
    if (report) record_error(p.err, DSA_DEVERR_BEHIND, r);
    return 0;
  }
  return len;
}

__device__ __forceinline__ int seq_written(const IndexParams& p, int seq) {
  return p.idx_written != nullptr ? p.idx_written[seq] : INT_MAX;
}

// Whether row r (length len, arena base rb) is well formed: the test
// row_len_checked makes, without the reporting.
__device__ __forceinline__ bool row_ok(const IndexParams& p, int len, int64_t rb, int64_t base,
                                       int written) {
  return len >= 0 && len <= p.max_len && rb == base && base >= 0 && base + len <= p.idx_tokens &&
         len <= written;
}

// Key tiles and arena base of group g (one thread).  The loads of every row
// are issued before any result is used (no store in between); the reasons
// for malformed rows are recorded in a second pass over them.
__device__ int group_tiles(const IndexParams& p, int g, bool report, int64_t& base) {
  const GroupRows gr = group_rows(p, g);
  base = p.idx_base[gr.seq_row0];
  const int written = seq_written(p, gr.seq);
  int m = 0;
  bool bad = false;
#pragma unroll 4
  for (int j = 0; j < gr.nrows; ++j) {
    const int len = p.seq_lens[gr.r0 + j];
    const bool ok = row_ok(p, len, p.idx_base[gr.r0 + j], base, written);
    m = max(m, ok ? len : 0);
    bad |= !ok;
  }
  if (report && bad)
    for (int j = 0; j < gr.nrows; ++j) row_len_checked(p, gr.r0 + j, base, written, true);
  return (m + kTileM - 1) / kTileM;
}

// Named barrier of the two scan warps.
__device__ __forceinline__ void scan_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kScanThreads) : "memory");
}
// Named barrier of warp 1 and the epilogue warps: the CTA's range and the
// TMEM address (written by tcgen05.alloc) are handed over here, with the
// tcgen05 fences on both sides of it.
__device__ __forceinline__ void tmem_sync() {
  asm volatile("bar.sync 3, %0;" ::"n"(32 + kEpiThreads) : "memory");
}

// Exclusive prefix of v over the scan threads (warps 0-1) in thread order,
// and their total.  Both warps must call it.
__device__ __forceinline__ long long scan_prefix(long long v, long long* scratch, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  scan_sync();
  const long long s0 = scratch[0], s1 = scratch[1];
  scan_sync();  // scratch may be reused
  total = s0 + s1;
  return (warp == 1 ? s0 : 0) + x - v;
}

// kDirect: a launch small enough for a few tiles per CTA in a single wave --
// CTA (x, y) scores tiles [x*dt, x*dt + dt) of group y (dt = direct_tiles,
// one stage each), needs no scan, and warp 0 loads the group's rows once,
// issues the tiles' copies and posts their record itself.
template <int D, bool kDirect>
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
  const int stages = p.stages;
  const int groups = (p.rows / p.rows_per_seq) * p.subs_per_seq;
  const long long ctas = gridDim.x, c = blockIdx.x;

  // ---------------------------------------------------------------- before the wait
  // Every input may be the output of the kernel before (the key arena and
  // gates of an indexer write, q and the head weights of a projection, row
  // metadata written on the device), so by default nothing is loaded before
  // grid_dep_wait().  When the caller declares the inputs complete before the
  // kernel before started (inputs_early), the wait moves to the epilogue's
  // first score store and to the exit: the loads, MMAs and score arithmetic
  // then overlap that kernel, and the scores buffer -- which a kernel before
  // may still read -- is written after it completes.  What overlaps the
  // kernel before in either case: barrier set-up, the
  // tensor map, and -- for a direct launch, or one of a single group, whose
  // split is known up to the row length -- L2 prefetches of the CTA's first
  // key tiles and of q (a
  // prefetch only warms L2, where the device's writes land, so it cannot make
  // a later load return a stale value; the arena base read for the address
  // may be stale, which only wastes the prefetch).
  const bool inputs_early = p.inputs_early != 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&ctl->tfull[a], 1);
      mbar_init(&ctl->tempty[a], kEpiThreads / 32);
    }
    mbar_init(&ctl->qready, kEpiThreads / 32);
    for (int k = 0; k < kSegRing; ++k) {
      mbar_init(&ctl->segfull[k], 1);
      mbar_init(&ctl->segfree[k], kEpiThreads / 32);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&kmap);
    // (With inputs_early the loads themselves go out right after the barrier
    // below; thread 0's prefetch still starts the first tiles' DRAM reads a
    // little sooner, which measured faster than skipping it.)
    if (kDirect || groups == 1) {
      const long long tg = (p.max_len + kTileM - 1) / kTileM;
      const long long b0 = kDirect ? static_cast<long long>(blockIdx.x) * p.direct_tiles : tg * c / ctas;
      const long long b1 = kDirect ? b0 + p.direct_tiles : tg * (c + 1) / ctas;
      const int64_t base_hint = *reinterpret_cast<const volatile int64_t*>(
          p.idx_base + group_rows(p, kDirect ? blockIdx.y : 0).seq_row0);
      for (long long t = b0; t < min(b1, b0 + stages); ++t) {
        const int64_t y = base_hint + t * kTileM;
        if (y >= 0 && y < p.idx_tokens)
#pragma unroll
          for (int sb = 0; sb < kSub; ++sb) tma_prefetch_l2_2d(&kmap, sb * 64, static_cast<int32_t>(y));
      }
    }
  }
  // A direct launch allocates TMEM now (it reads no input); a persistent one
  // once the scan has shown that the CTA has tiles.
  if (kDirect && warp == 1) {
    tmem_alloc(&ctl->tmem_base, p.tmem_cols);
    tmem_relinquish();
  }
  if ((kDirect || groups == 1) && !inputs_early) {
    const GroupRows gr = group_rows(p, kDirect ? blockIdx.y : 0);
    const float* qsrc = p.q_idx + static_cast<int64_t>(gr.r0) * p.heads * D;
    for (int off = threadIdx.x * 32; off < gr.nrows * p.heads * D; off += kThreads * 32)
      prefetch_l2(qsrc + off);
    if (threadIdx.x < gr.nrows) prefetch_l2(p.seq_lens + gr.r0 + threadIdx.x);
  }
  // The barriers are initialised before any warp can arrive on or wait for
  // one: the roles below start without a CTA-wide barrier between them.
  __syncthreads();
  if (!inputs_early) grid_dep_wait();

  // ---------------------------------------------------------------- this CTA's range
  // Warps 0-1 find the range -- pass 1: T = sum of T_g (CTA 0 records the
  // malformed rows); pass 2: the group holding tile `begin` -- then warp 1
  // allocates TMEM and meets the epilogue warps at tmem_sync().  Groups are taken kScanThreads at a
  // time, one per thread; the first kScanRegs rounds keep T_g and the base
  // for pass 2.  Meanwhile the epilogue warps build the q operand of a launch
  // with a single group, which needs no scan to be known.
  long long my_tiles = 0;
  uint32_t tmem_base = 0;
  if (warp < 2) {
   if constexpr (kDirect) {
    if (warp == 0) {
      // The group's rows, one per lane; every lane's loads issued together.
      const int g = blockIdx.y, t0 = blockIdx.x * p.direct_tiles;
      const GroupRows gr = group_rows(p, g);
      const int64_t base = p.idx_base[gr.seq_row0];
      const int written = seq_written(p, gr.seq);
      const bool has_row = lane < gr.nrows;
      const int len_raw = has_row ? p.seq_lens[gr.r0 + lane] : 0;
      const int64_t rb = has_row ? p.idx_base[gr.r0 + lane] : base;
      const bool row_good = row_ok(p, len_raw, rb, base, written);
      const int len = has_row && row_good ? len_raw : 0;
      if (has_row && !row_good && t0 == 0) row_len_checked(p, gr.r0 + lane, base, written, true);
      int m = len;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const int tg = (m + kTileM - 1) / kTileM;
      my_tiles = max(0, min(p.direct_tiles, tg - t0));
      if (my_tiles > 0) {
        Seg& sg = ctl->seg[0];
        sg.row_len[lane] = len;
        if (lane == 0) {
          const uint64_t policy = l2_policy_evict_first();
          for (int j = 0; j < my_tiles; ++j) {
            mbar_arrive_expect_tx(&ctl->full[j], kStageBytes);
            const int32_t y = static_cast<int32_t>(base + static_cast<int64_t>(t0 + j) * kTileM);
#pragma unroll
            for (int sb = 0; sb < kSub; ++sb)
              tma_load_2d(stage_base + j * kStageBytes + sb * (kTileM * 128), &kmap, &ctl->full[j],
                          sb * 64, y, policy);
          }
          sg.base = base;
          sg.r0 = gr.r0;
          sg.nrows = gr.nrows;
          sg.t_first = t0;
          sg.ntiles = static_cast<int>(my_tiles);
          sg.max_len = m;
          ctl->g0 = g;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->segfull[0]);
      }
      if (lane == 0) ctl->my_tiles = my_tiles;
    }
    scan_sync();  // my_tiles, g0
    my_tiles = ctl->my_tiles;
   } else {
    const int st = threadIdx.x;
    const bool report = blockIdx.x == 0;
    int tg_keep[kScanRegs];
    int64_t base_keep[kScanRegs];
    long long mine = 0;
#pragma unroll
    for (int k = 0; k < kScanRegs; ++k) {
      const int g = k * kScanThreads + st;
      base_keep[k] = 0;
      tg_keep[k] = g < groups ? group_tiles(p, g, report, base_keep[k]) : 0;
      mine += tg_keep[k];
    }
    for (int g = kScanRegs * kScanThreads + st; g < groups; g += kScanThreads) {
      int64_t b;
      mine += group_tiles(p, g, report, b);
    }
    long long total;
    scan_prefix(mine, ctl->scan, total);
    const long long begin = total * c / ctas, end = total * (c + 1) / ctas;
    my_tiles = end > begin ? end - begin : 0;
    if (my_tiles > 0) {
      long long running = 0;
      for (int k = 0; k * kScanThreads < groups; ++k) {  // uniform trip count
        const int g = k * kScanThreads + st;
        int v = 0;
        int64_t b = 0;
#pragma unroll
        for (int kk = 0; kk < kScanRegs; ++kk)
          if (kk == k) {
            v = tg_keep[kk];
            b = base_keep[kk];
          }
        if (k >= kScanRegs && g < groups) v = group_tiles(p, g, false, b);
        long long round_total;
        const long long ex = running + scan_prefix(v, ctl->scan, round_total);
        if (v > 0 && ex <= begin && begin < ex + v) {
          ctl->g0 = g;
          ctl->t0 = static_cast<int>(begin - ex);
          ctl->tg0 = v;
          ctl->base0 = b;
        }
        running += round_total;
        if (running > begin) break;  // uniform: every scan thread holds the same total
      }
    }
    if (st == 0) ctl->my_tiles = my_tiles;
    scan_sync();  // g0 / t0 / tg0 / base0 / my_tiles
   }
    if (warp == 1) {
      if (!kDirect && my_tiles > 0) {
        tmem_alloc(&ctl->tmem_base, p.tmem_cols);
        tmem_relinquish();
      }
      tc_fence_before();
      tmem_sync();  // every path of warp 1 and of the epilogue warps passes it once
      tc_fence_after();
      if (my_tiles > 0) tmem_base = ctl->tmem_base;
    }
  }

  // ---------------------------------------------------------------- roles
  if (kDirect && warp == 0 && my_tiles > 0) {
    // The CTA's tiles went out with its record: never leave with one in flight.
    if (lane == 0)
      for (int j = 0; j < my_tiles; ++j) mbar_wait(&ctl->full[j], 0, kDrainWaitNs);
  } else if (!kDirect && warp == 0 && my_tiles > 0) {
    // ============================================================ segments + TMA
    uint64_t policy = 0;
    if (lane == 0) policy = l2_policy_evict_first();
    int g = ctl->g0, t0 = ctl->t0;
    long long remaining = my_tiles;
    int k = 0, issued = 0;
    bool ok = true;
    // Segment 0's first tiles go out at once: the scan gave its group's base
    // and tile count, so they need no load; its rows are checked meanwhile.
    const int pre = static_cast<int>(min(static_cast<long long>(min(ctl->tg0 - t0, stages)), remaining));
    if (lane == 0) {
      const int64_t base0 = ctl->base0;
      for (; issued < pre; ++issued) {
        const int32_t y = static_cast<int32_t>(base0 + static_cast<int64_t>(t0 + issued) * kTileM);
        mbar_arrive_expect_tx(&ctl->full[issued], kStageBytes);
#pragma unroll
        for (int sb = 0; sb < kSub; ++sb)
          tma_load_2d(stage_base + issued * kStageBytes + sb * (kTileM * 128), &kmap,
                      &ctl->full[issued], sb * 64, y, policy);
      }
    }
    while (ok && remaining > 0 && g < groups) {
      // The group's rows, one per lane (at most 32 rows per group); every
      // lane's loads are issued before any is used.
      const GroupRows gr = group_rows(p, g);
      const int64_t base = p.idx_base[gr.seq_row0];
      const int written = seq_written(p, gr.seq);
      const bool has_row = lane < gr.nrows;
      const int len_raw = has_row ? p.seq_lens[gr.r0 + lane] : 0;
      const int64_t rb = has_row ? p.idx_base[gr.r0 + lane] : base;
      const int len = has_row && row_ok(p, len_raw, rb, base, written) ? len_raw : 0;
      int m = len;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const int tg = (m + kTileM - 1) / kTileM;
      if (tg <= t0) {  // a group with no tiles (never the first: it holds tile `begin`)
        ++g;
        t0 = 0;
        continue;
      }
      const int n = static_cast<int>(min(static_cast<long long>(tg - t0), remaining));
      // q rows and head weights of the segment into L2 for the epilogue's build.
      const int nreal = gr.nrows * p.heads;
      const float* qsrc = p.q_idx + static_cast<int64_t>(gr.r0) * p.heads * D;
      if (k > 0) {  // segment 0's operand is being built already
        for (int off = lane * 32; off < nreal * D; off += 32 * 32) prefetch_l2(qsrc + off);
        if (lane * 32 < nreal) prefetch_l2(p.head_w + static_cast<int64_t>(gr.r0) * p.heads + lane * 32);
      }
      const int slot = k % kSegRing;
      int w_ok = 1;
      if (lane == 0 && k >= kSegRing)
        w_ok = mbar_wait(&ctl->segfree[slot], ((k / kSegRing) - 1) & 1, p.wait_ns) ? 1 : 0;
      w_ok = __shfl_sync(0xFFFFFFFFu, w_ok, 0);
      if (!w_ok) {
        if (lane == 0) set_abort(ctl, p.err, gr.r0);
        break;
      }
      Seg& sg = ctl->seg[slot];
      if (lane < kMaxSubRows) sg.row_len[lane] = len;
      if (lane == 0) {
        sg.base = base;
        sg.r0 = gr.r0;
        sg.nrows = gr.nrows;
        sg.t_first = t0;
        sg.ntiles = n;
        sg.max_len = m;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->segfull[slot]);
        for (int i = k == 0 ? pre : 0; i < n; ++i, ++issued) {
          if (aborted(ctl)) {
            ok = false;
            break;
          }
          const int s = issued % stages;
          if (issued >= stages && !mbar_wait(&ctl->empty[s], ((issued / stages) - 1) & 1, p.wait_ns)) {
            set_abort(ctl, p.err, gr.r0);
            ok = false;
            break;
          }
          uint8_t* dst = stage_base + s * kStageBytes;
          const int32_t y = static_cast<int32_t>(base + static_cast<int64_t>(t0 + i) * kTileM);
          mbar_arrive_expect_tx(&ctl->full[s], kStageBytes);
#pragma unroll
          for (int sb = 0; sb < kSub; ++sb)
            tma_load_2d(dst + sb * (kTileM * 128), &kmap, &ctl->full[s], sb * 64, y, policy);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      remaining -= n;
      ++k;
      ++g;
      t0 = 0;
    }
    // Never leave with a copy in flight: wait (bounded) for the last loads.
    issued = __shfl_sync(0xFFFFFFFFu, issued, 0);
    if (lane == 0)
      for (int i = max(0, issued - stages); i < issued; ++i)
        mbar_wait(&ctl->full[i % stages], (i / stages) & 1, kDrainWaitNs);
  } else if (warp == 1 && my_tiles > 0) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTileM, npad);
      const uint32_t a0 = smem_u32(stage_base), bh = smem_u32(b_hi), bl = smem_u32(b_lo);
      long long done = 0;
      int i = 0;
      bool ok = true;
      for (int k = 0; ok && done < my_tiles; ++k) {
        const int slot = k % kSegRing;
        if (aborted(ctl) || !mbar_wait(&ctl->segfull[slot], (k / kSegRing) & 1, p.wait_ns) ||
            !mbar_wait(&ctl->qready, k & 1, p.wait_ns)) {
          if (!aborted(ctl)) set_abort(ctl, p.err, -1);
          break;
        }
        const int n = ctl->seg[slot].ntiles;
        for (int j = 0; j < n; ++j, ++i) {
          const int s = i % stages, a = i & 1;
          if (aborted(ctl) || !mbar_wait(&ctl->full[s], (i / stages) & 1, p.wait_ns) ||
              (i >= 2 && !mbar_wait(&ctl->tempty[a], ((i >> 1) - 1) & 1, p.wait_ns))) {
            if (!aborted(ctl)) set_abort(ctl, p.err, -1);
            ok = false;
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
        done += n;
      }
      // Every MMA issued by this thread is complete before TMEM is released.
      umma_commit(&ctl->drain);
      mbar_wait(&ctl->drain, 0, kDrainWaitNs);
    }
  } else if (warp >= 2) {
    // ============================================================ q build + epilogue
    // Every epilogue warp passes the same named barriers in the same order
    // whatever happens (a timed-out wait only makes the warp skip work), and
    // they leave the segment loop together.
    const int et = threadIdx.x - 64;            // 0..127
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. = tokens
    const int lane_tok = quarter * 32 + lane;
    const int heads = p.heads;
    const int cols_per_row = (heads % 16 == 0) ? heads : npad;  // heads%16 != 0 -> one row
    const int vec_per_row = D / 8;
    const int nvec = npad * vec_per_row;
    constexpr int kBatch = 8;
    constexpr int kWPer = 256 / kEpiThreads;  // head-weight columns per thread (npad <= 256)
    // B operand of the group whose rows start at r0: q split into bf16 hi +
    // lo, in the 128-byte-swizzled K-major layout the MMA descriptor expects
    // (row n at n*128 B inside a 64-element sub-tile, 16-byte chunk c stored
    // at chunk c ^ (n % 8)); rows past the group's real ones are zero.  The
    // head weights are loaded with the first batch of q.  Ends with this
    // warp's arrival on qready.
    auto build_q = [&](int r0, int nrows) {
      const int nreal = nrows * heads;
      const float* qsrc = p.q_idx + static_cast<int64_t>(r0) * heads * D;
      float wv[kWPer];
#pragma unroll
      for (int e = 0; e < kWPer; ++e) {
        const int col = et + e * kEpiThreads;
        wv[e] = col < nreal ? p.head_w[static_cast<int64_t>(r0) * heads + col] : 0.0f;
      }
      for (int v0 = et; v0 < nvec; v0 += kBatch * kEpiThreads) {
        float4 u[kBatch][2];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = v0 + b * kEpiThreads;
          const int row = v / vec_per_row, c8 = v % vec_per_row;
          if (v < nvec && row < nreal) {
            const float4* src = reinterpret_cast<const float4*>(qsrc + static_cast<int64_t>(row) * D + c8 * 8);
            u[b][0] = ld_dep_f4(src);
            u[b][1] = ld_dep_f4(src + 1);
          } else {
            u[b][0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            u[b][1] = u[b][0];
          }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int v = v0 + b * kEpiThreads;
          if (v >= nvec) break;
          const int row = v / vec_per_row, c8 = v % vec_per_row;
          const float x[8] = {u[b][0].x, u[b][0].y, u[b][0].z, u[b][0].w,
                              u[b][1].x, u[b][1].y, u[b][1].z, u[b][1].w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(x[2 * e]);
            const __nv_bfloat16 h1 = __float2bfloat16_rn(x[2 * e + 1]);
            const float r0f = x[2 * e] - __bfloat162float(h0);
            const float r1f = x[2 * e + 1] - __bfloat162float(h1);
            hi[e] = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
            lo[e] = pack_bf16x2(r0f, r1f);
          }
          const int sb = (c8 * 8) / 64, chunk = c8 & 7;
          const uint32_t off = sb * (npad * 128) + row * 128 + ((chunk ^ (row & 7)) * 16);
          *reinterpret_cast<uint4*>(b_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(b_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
#pragma unroll
      for (int e = 0; e < kWPer; ++e) {
        const int col = et + e * kEpiThreads;
        if (col < npad) w_s[col] = wv[e];
      }
      fence_proxy_async_smem();  // generic-proxy smem writes -> visible to the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->qready);
    };
    // Segment 0's operand: right away when the group is known without a scan
    // (a direct launch, or a single group), otherwise as soon as the scan has
    // named it; either way it overlaps the row checks and the first key loads.
    const bool early = kDirect || groups == 1;  // the group is known without a scan
    if (early) {
      const GroupRows gr = group_rows(p, kDirect ? blockIdx.y : 0);
      build_q(gr.r0, gr.nrows);
    }
    // The range and the TMEM address from warps 0-1 (the scan has no waits,
    // so warp 1 always gets here).
    tc_fence_before();
    tmem_sync();
    tc_fence_after();
    my_tiles = ctl->my_tiles;
    if (my_tiles > 0) tmem_base = ctl->tmem_base;
    if (my_tiles > 0 && !early) {
      const GroupRows gr = group_rows(p, ctl->g0);
      build_q(gr.r0, gr.nrows);
    }
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    bool waited = !inputs_early;
    long long done = 0;
    int i = 0;        // tiles consumed by this CTA so far (TMEM buffer and phase)
    bool ok = true;
    for (int k = 0;; ++k) {
      const int slot = k % kSegRing;
      // One lane polls; the warp then continues together.
      int w = 0;
      if (done < my_tiles && ok) {
        if (lane == 0) w = mbar_wait(&ctl->segfull[slot], (k / kSegRing) & 1, p.wait_ns) ? 1 : 2;
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (w == 2 && lane == 0) set_abort(ctl, p.err, -1);
      }
      // Leave together when this CTA is done or any warp failed.  The barrier
      // also orders the previous segment's reads of w_s before its rewrite.
      if (epi_sync_or(w != 1)) break;
      const Seg& sg = ctl->seg[slot];
      const int r0 = sg.r0, nrows = sg.nrows, n = sg.ntiles, t_first = sg.t_first;
      const int max_len_group = sg.max_len;
      const int64_t base = sg.base;
      // Later segments: the previous segment's MMAs are complete (this warp
      // consumed its last accumulator), so the operand can be rewritten.
      if (k > 0) build_q(r0, nrows);
      epi_sync();                // w_s complete before any warp reads it

      // Each tile's gate is loaded one tile ahead, so the load's DRAM latency
      // hides behind the TMA and the MMAs (plain loads: the gates may come
      // from the kernel before, which the wait at the top has ordered unless
      // the caller declared them complete before it).
      auto load_gate = [&](int j) {
        const int t = (t_first + j) * kTileM + lane_tok;
        return (j < n && t < max_len_group) ? p.gate[base + t] : static_cast<uint16_t>(0);
      };
      uint16_t g_next = load_gate(0);
      for (int j = 0; j < n && ok; ++j, ++i) {
        const int a = i & 1;
        const int t = (t_first + j) * kTileM + lane_tok;
        const float gt = __bfloat162float(__ushort_as_bfloat16(g_next));
        g_next = load_gate(j + 1);
        int wok = 1;
        if (lane == 0) wok = mbar_wait(&ctl->tfull[a], (i >> 1) & 1, p.wait_ns) ? 1 : 0;
        wok = __shfl_sync(0xFFFFFFFFu, wok, 0);
        if (!wok) {
          if (lane == 0) set_abort(ctl, p.err, r0);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = lane_addr + a * npad;
        for (int jr = 0; jr < nrows; ++jr) {
          // Columns in ascending order, 32 per TMEM read (16 at an odd end).
          // Columns past the real ones hold 0 (zero q rows) with weight 0, so
          // they add +-0 and leave the sum as it is (it is never -0).
          float sum = 0.0f;
          const int c_begin = jr * cols_per_row, c_end = c_begin + cols_per_row;
          int c0 = c_begin;
          for (; c0 + 32 <= c_end; c0 += 32) {
            float v[32];
            tmem_load32(acc + c0, v);
            const float4* w4 = reinterpret_cast<const float4*>(w_s + c0);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 w = w4[e];
              sum = fmaf(w.x, fmaxf(v[4 * e], 0.0f), sum);
              sum = fmaf(w.y, fmaxf(v[4 * e + 1], 0.0f), sum);
              sum = fmaf(w.z, fmaxf(v[4 * e + 2], 0.0f), sum);
              sum = fmaf(w.w, fmaxf(v[4 * e + 3], 0.0f), sum);
            }
          }
          if (c0 < c_end) {
            float v[16];
            tmem_load16(acc + c0, v);
            const float4* w4 = reinterpret_cast<const float4*>(w_s + c0);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 w = w4[e];
              sum = fmaf(w.x, fmaxf(v[4 * e], 0.0f), sum);
              sum = fmaf(w.y, fmaxf(v[4 * e + 1], 0.0f), sum);
              sum = fmaf(w.z, fmaxf(v[4 * e + 2], 0.0f), sum);
              sum = fmaf(w.w, fmaxf(v[4 * e + 3], 0.0f), sum);
            }
          }
          if (t < sg.row_len[jr]) {
            if (!waited) {  // (inputs_early) the first store waits for the kernel before
              grid_dep_wait();
              waited = true;
            }
            p.scores[static_cast<int64_t>(r0 + jr) * p.max_len + t] = gt * sum;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->tempty[a]);
        if (__shfl_sync(0xFFFFFFFFu, aborted(ctl) ? 1 : 0, 0)) {
          ok = false;
          break;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->segfree[slot]);
      done += n;
    }
  }

  // ---------------------------------------------------------------- teardown
  // (inputs_early) No CTA completes before the kernel before has: whatever
  // waits for this kernel also waits for that one.
  if (inputs_early) grid_dep_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 1 && (kDirect || my_tiles > 0)) {
    tc_fence_after();
    tmem_dealloc(kDirect ? ctl->tmem_base : tmem_base, p.tmem_cols);
  }
}

}  // namespace

void plan_index_scores(IndexParams& p, int num_sms) {
  const uint32_t stage_bytes = kTileM * p.dim * 2;
  const uint32_t b_bytes = 2u * p.npad * p.dim * 2;
  const uint32_t fixed = b_bytes + p.npad * 4 + sizeof(IndexCtl) + 1024;  // + alignment slack
  const uint32_t two_per_sm = 113u * 1024u, one_per_sm = 226u * 1024u;
  int stages = 0, per_sm = 1;
  if (fixed + 2 * stage_bytes <= two_per_sm) {
    stages = static_cast<int>((two_per_sm - fixed) / stage_bytes);
    per_sm = 2;
  } else {
    stages = static_cast<int>((one_per_sm - fixed) / stage_bytes);
  }
  stages = stages > 4 ? 4 : stages;
  if (stages < 1) stages = 1;

  // A launch whose tiles fit one wave even at the longest possible rows runs
  // direct (one tile per CTA, one stage); any other one persistent CTAs, one
  // wave of them.
  const int64_t tiles_max = (static_cast<int64_t>(p.max_len) + kTileM - 1) / kTileM;
  const int64_t groups = static_cast<int64_t>(p.rows / p.rows_per_seq) * p.subs_per_seq;
  const int64_t wave = static_cast<int64_t>(per_sm) * num_sms;
  p.direct = (tiles_max * groups <= wave && groups <= 65535) ? 1 : 0;
  p.direct_tiles = kDirectTiles;
  if (p.direct) stages = kDirectTiles;
  p.stages = stages;
  p.smem_bytes = fixed + stages * stage_bytes;
  int64_t ctas = wave;
  if (ctas > tiles_max * groups) ctas = tiles_max * groups;
  p.ctas = static_cast<int32_t>(ctas < 1 ? 1 : ctas);

  uint32_t cols = 32;
  while (cols < 2u * p.npad) cols <<= 1;
  p.tmem_cols = cols;
}

cudaError_t launch_index_scores(const IndexParams& p, const CUtensorMap& kmap,
                                cudaStream_t stream) {
  const int64_t groups = static_cast<int64_t>(p.rows / p.rows_per_seq) * p.subs_per_seq;
  if (groups <= 0 || p.max_len <= 0) return cudaSuccess;
  if (groups > INT_MAX / 2) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  auto kernel = p.direct ? (p.dim == 64 ? index_scores_kernel<64, true> : index_scores_kernel<128, true>)
                        : (p.dim == 64 ? index_scores_kernel<64, false> : index_scores_kernel<128, false>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  const int64_t tiles_max = (static_cast<int64_t>(p.max_len) + kTileM - 1) / kTileM;
  cfg.gridDim = p.direct ? dim3(static_cast<unsigned>((tiles_max + p.direct_tiles - 1) / p.direct_tiles),
                                static_cast<unsigned>(groups), 1)
                         : dim3(static_cast<unsigned>(p.ctas), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, kmap, p);
}

}  // namespace dsa
