// mla_decode_cluster.cu -- S3: absorbed NoPE MLA gather-attend, one
// thread-block cluster per (row, 64-head group).
//
// "glm5next_dsa/layer.rs": module header trap 4 (Q arrives absorbed into the
// 512-wide latent space; the kernel dots Q against the latent directly),
// attend_rows (one launch for all rows, each with its own selection row,
// seq_len and block-table row; K and V are the same latent pool), decode_k
// (slot = block * block_size + pos % block_size).  Per row and head:
//     z_j = sm_scale * kv_scale * (Q . e4m3(latent_j)),  p = softmax(z)
//     out = kv_scale * sum_j p_j e4m3(latent_j),  lse = log sum_j exp(z_j)
//
// The selection of a row is cut into n <= 16 equal splits (n depends only on
// topk and the device, so a row's arithmetic never depends on the other rows
// of the call).  The n CTAs of one (row, 64 heads) form a cluster.  Each CTA
// (16 warps) streams its split's latent rows in 32-token tiles (16-byte
// cp.async gathers, 3-stage ring), widens FP8 to f16 in shared memory once for
// all 64 heads (one exact cvt per pair) and runs S = Q K^T and
// O = alpha O + P V on f16 tensor-core MMAs with FP32 accumulation and an
// online softmax.  Q is scaled per head by a power of two so its bf16 values
// are exact in f16; heads past the row's head count are zero and never
// written.  The n partial (m, l, O) then merge through distributed shared
// memory in fixed split order; nothing goes through global memory.
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kMT = 4;               // 16-head m-tiles per CTA
constexpr int kHG = 16 * kMT;        // heads per CTA
constexpr int kTok = 32;             // tokens per tile
constexpr int kStages = 3;           // cp.async ring depth
constexpr int kMaxSplits = 16;       // cluster size bound
constexpr int kRowB = 1040;          // bytes per f16 row of 512 (+16 pad: conflict-free ldmatrix)
constexpr int kPRowB = (kTok + 8) * 2;  // bytes per f16 row of P
constexpr int kChunk = 512;          // selection entries whose slots are resolved together
constexpr int kTilesPerChunk = kChunk / kTok;

struct Smem {
  uint8_t q[kHG * kRowB];
  uint8_t kv[kTok * kRowB];
  uint8_t stage[kStages][kTok * 512];
  float s[kHG][kTok + 1];
  uint8_t pmat[kHG * kPRowB];
  int64_t slot[kChunk];
  int8_t valid[kStages][kTok];
  float m[kHG], l[kHG], alpha[kHG], qexp[kHG];
};
// The merge reuses the q + kv + stage region for the partial O [64][512] fp32.
static_assert(sizeof(float) * kHG * 512 <= kHG * kRowB + kTok * kRowB + kStages * kTok * 512,
              "partial O does not fit");

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
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
__device__ __forceinline__ uint32_t remote_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// Volatile (ordered after the cluster barrier) but without a memory clobber,
// so independent remote loads are issued back to back.
__device__ __forceinline__ float ld_remote_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float4 ld_remote_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_cluster_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int hg = blockIdx.y, r = blockIdx.z;
  const uint32_t split = cluster_rank();
  const int nsplit = p.splits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split_len = p.split_len;
  const int j0 = static_cast<int>(split) * split_len;
  const int nj = max(0, min(split_len, p.topk - j0));
  const bool report = hg == 0;
  const int head0 = hg * kHG;
  const int nheads = min(kHG, p.heads - head0);

  grid_dep_wait();  // the selection comes from the kernel before
  grid_dep_launch();
  int len = p.rows.seq_lens[r];
  if (len < 0) {
    if (report && split == 0 && tid == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }
  const int32_t* bt = p.rows.block_table + static_cast<int64_t>(r) * p.rows.bt_stride;
  const int bs = p.rows.block_size;
  const int32_t* sel_row = p.sel + static_cast<int64_t>(r) * p.topk + j0;
  const int ntiles = (nj + kTok - 1) / kTok;

  // Physical slots of selection entries [ch*kChunk, (ch+1)*kChunk) of this
  // split (-1: padding or invalid); out-of-range entries are recorded, not read.
  auto resolve_chunk = [&](int ch) {
    for (int i = tid; i < kChunk; i += kThreads) {
      const int j = ch * kChunk + i;
      int64_t slot = -1;
      if (j < nj) {
        const int idx = __ldg(sel_row + j);
        if (idx != -1) {
          if (idx < 0 || idx >= len) {
            if (report) record_error(p.err, DSA_DEVERR_SELECT, r);
          } else {
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
      sm.slot[i] = slot;
    }
  };
  // Gather one tile of selected latent rows into a stage: 32 tokens x 32
  // chunks of 16 B, two chunks per thread.
  auto issue_tile = [&](int tile, int buf) {
#pragma unroll
    for (int j = 0; j < kTok * 32 / kThreads; ++j) {
      const int c = tid + j * kThreads;
      const int tok = c >> 5, k = c & 31;
      const int i = tile * kTok + tok;
      const int64_t slot = i < nj ? sm.slot[i % kChunk] : -1;
      if (k == 0) sm.valid[buf][tok] = slot >= 0 ? 1 : 0;
      const uint8_t* src = slot >= 0 ? p.pool + slot * 512 + k * 16 : p.pool;
      cp_async16(&sm.stage[buf][tok * 512 + k * 16], src, slot >= 0 ? 16u : 0u);
    }
    cp_async_commit();
  };

  resolve_chunk(0);
  __syncthreads();
  for (int t = 0; t < kStages - 1; ++t) {
    if (t < ntiles) issue_tile(t, t);
    else cp_async_commit();  // keep the group count uniform
  }

  // Q -> f16, each head scaled by 2^(14 - e) with max|q_h| < 2^e, so every
  // bf16 value is exactly representable (f16 carries 11 significant bits).
  // 8 threads per head, 64 elements each; heads past the row's count are 0.
  {
    const int h = tid >> 3, part = tid & 7;
    const bool real = h < nheads;
    const uint16_t* qsrc = p.q + (static_cast<int64_t>(r) * p.heads + head0 + h) * 512 + part * 64;
    uint4 raw[8];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)  // all eight loads in flight before any is used
      raw[j] = real ? __ldg(reinterpret_cast<const uint4*>(qsrc) + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    int e = 0;
    if (amax > 0.0f) frexpf(amax, &e);  // amax < 2^e
    const int sh = max(-100, min(100, 14 - e));
    const float scale = ldexpf(1.0f, sh);
    if (part == 0) {
      sm.qexp[h] = static_cast<float>(sh);
      sm.m[h] = -INFINITY;
      sm.l[h] = 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
      uint32_t o4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o4[i] = pack_f16x2(__uint_as_float(w[i] << 16) * scale,
                           __uint_as_float(w[i] & 0xFFFF0000u) * scale);
      *reinterpret_cast<uint4*>(sm.q + h * kRowB + (part * 64 + j * 8) * 2) =
          make_uint4(o4[0], o4[1], o4[2], o4[3]);
    }
  }

  // PV accumulators: warp w owns latent dims 32w .. 32w+31 for all 64 heads.
  float o[kMT][4][4];
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.0f;
  const float base_scale = p.sm_scale * p.kv_scale * 1.4426950408889634f;
  const int g = lane >> 2, t2 = (lane & 3) * 2;
  const int s_mt = warp & 3, s_nt = warp >> 2;  // S-phase tile of this warp

  for (int it = 0; it < ntiles; ++it) {
    const int buf = it % kStages;
    const int next = it + kStages - 1;
    if (next < ntiles) {
      if (next % kTilesPerChunk == 0) {  // first tile of a new chunk of entries
        __syncthreads();
        resolve_chunk(next / kTilesPerChunk);
        __syncthreads();
      }
      issue_tile(next, next % kStages);
    } else {
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();

    // FP8 -> f16 (exact) into the padded latent tile, once for all heads.
    const uint8_t* st = sm.stage[buf];
#pragma unroll
    for (int j = 0; j < kTok * 32 / kThreads; ++j) {
      const int c = tid + j * kThreads;
      const int tok = c >> 5, k = c & 31;
      const uint4 raw = *reinterpret_cast<const uint4*>(st + tok * 512 + k * 16);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t cv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cv[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] & 0xFFFFu));
        cv[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] >> 16));
      }
      uint4* dst = reinterpret_cast<uint4*>(sm.kv + tok * kRowB + k * 32);
      dst[0] = make_uint4(cv[0], cv[1], cv[2], cv[3]);
      dst[1] = make_uint4(cv[4], cv[5], cv[6], cv[7]);
    }
    __syncthreads();

    // S = Q K^T: warp w computes heads 16*(w%4) .. +15 against tokens
    // 8*(w/4) .. +7, four independent accumulator chains over the 32 K steps.
    {
      float acc[4][4] = {};
      const uint32_t a_addr = smem_u32(sm.q) +
                              (s_mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kRowB +
                              (lane >> 4) * 16;
      const uint32_t b_addr =
          smem_u32(sm.kv) + (s_nt * 8 + (lane & 7)) * kRowB + ((lane >> 3) & 1) * 16;
      // Fragments are loaded two K steps ahead of the MMA that uses them.
      uint32_t af[3][4], bf[3][2];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        ldsm_x4(a_addr + kk * 32, af[kk][0], af[kk][1], af[kk][2], af[kk][3]);
        ldsm_x2(b_addr + kk * 32, bf[kk][0], bf[kk][1]);
      }
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        if (kk + 2 < 32) {
          const int nb = (kk + 2) % 3;
          ldsm_x4(a_addr + (kk + 2) * 32, af[nb][0], af[nb][1], af[nb][2], af[nb][3]);
          ldsm_x2(b_addr + (kk + 2) * 32, bf[nb][0], bf[nb][1]);
        }
        const int cb = kk % 3;
        mma_f16_16816(acc[kk & 3], af[cb][0], af[cb][1], af[cb][2], af[cb][3], bf[cb][0], bf[cb][1]);
      }
      const int h0 = s_mt * 16 + g;
      const float sc0 = base_scale * exp2f(-sm.qexp[h0]);
      const float sc1 = base_scale * exp2f(-sm.qexp[h0 + 8]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
        const int h = h0 + (e >> 1) * 8, tok = s_nt * 8 + t2 + (e & 1);
        const bool ok = it * kTok + tok < nj && sm.valid[buf][tok];
        sm.s[h][tok] = ok ? v * ((e >> 1) ? sc1 : sc0) : -INFINITY;
      }
    }
    __syncthreads();

    // Online softmax (base 2): 8 threads per head, 4 tokens each.
    {
      const int h = tid >> 3, q4 = (tid & 7) * 4;
      float v[4], mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[i] = sm.s[h][q4 + i];
        mx = fmaxf(mx, v[i]);
      }
#pragma unroll
      for (int o2 = 1; o2 < 8; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o2));
      const float m_old = sm.m[h];
      const float m_new = fmaxf(m_old, mx);
      float alpha = 1.0f, psum = 0.0f, pv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (m_new != -INFINITY) {
        alpha = exp2f(m_old - m_new);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pv[i] = exp2f(v[i] - m_new);
          psum += pv[i];
        }
      }
#pragma unroll
      for (int o2 = 1; o2 < 8; o2 <<= 1) psum += __shfl_xor_sync(0xFFFFFFFFu, psum, o2);
      uint32_t* prow = reinterpret_cast<uint32_t*>(sm.pmat + h * kPRowB + q4 * 2);
      prow[0] = pack_f16x2(pv[0], pv[1]);
      prow[1] = pack_f16x2(pv[2], pv[3]);
      if ((tid & 7) == 0) {
        sm.l[h] = sm.l[h] * alpha + psum;
        sm.m[h] = m_new;
        sm.alpha[h] = alpha;
      }
    }
    __syncthreads();

    // O = alpha O + P V on this warp's 32 latent dims.
    {
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt) {
        const float al0 = sm.alpha[mt * 16 + g], al1 = sm.alpha[mt * 16 + g + 8];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          o[mt][nt][0] *= al0;
          o[mt][nt][1] *= al0;
          o[mt][nt][2] *= al1;
          o[mt][nt][3] *= al1;
        }
      }
      const uint32_t pbase = smem_u32(sm.pmat), kvbase = smem_u32(sm.kv);
#pragma unroll
      for (int ks = 0; ks < kTok / 16; ++ks) {
        // Every fragment of this K step is requested before the first MMA.
        uint32_t b[4][2], a[kMT][4];
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int d0 = warp * 32 + np * 16;
          ldsm_x4_trans(kvbase + (ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kRowB +
                            (d0 + (lane >> 4) * 8) * 2,
                        b[2 * np][0], b[2 * np][1], b[2 * np + 1][0], b[2 * np + 1][1]);
        }
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
          ldsm_x4(pbase + (mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kPRowB + ks * 32 +
                      (lane >> 4) * 16,
                  a[mt][0], a[mt][1], a[mt][2], a[mt][3]);
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
            mma_f16_16816(o[mt][nt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], b[nt][0], b[nt][1]);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // the q / kv / stage region is reused for the partial O below

  // ---- this split's partial (m, l, unnormalised O) in shared memory
  float* part = reinterpret_cast<float*>(sm.q);
#pragma unroll
  for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int d = warp * 32 + nt * 8 + t2;
      const int h = mt * 16 + g;
      *reinterpret_cast<float2*>(part + h * 512 + d) = make_float2(o[mt][nt][0], o[mt][nt][1]);
      *reinterpret_cast<float2*>(part + (h + 8) * 512 + d) = make_float2(o[mt][nt][2], o[mt][nt][3]);
    }
  cluster_sync();

  // ---- merge: CTA `split` finishes heads split, split+n, ... (128 threads per
  // head, 4 dims each) over all n splits in split order.
  const int per_cta = (kHG + nsplit - 1) / nsplit;
  for (int item = tid; item < per_cta * 128; item += kThreads) {
    const int h = static_cast<int>(split) + (item >> 7) * nsplit;
    const int d4 = item & 127;
    if (h >= nheads) continue;
    // All remote reads of this item are issued before any is used.
    float mc[kMaxSplits], lc[kMaxSplits];
    float4 vc[kMaxSplits];
#pragma unroll
    for (int c = 0; c < kMaxSplits; ++c)
      if (c < nsplit) {
        mc[c] = ld_remote_f32(remote_addr(&sm.m[h], c));
        lc[c] = ld_remote_f32(remote_addr(&sm.l[h], c));
        vc[c] = ld_remote_f32x4(remote_addr(part + h * 512 + d4 * 4, c));
      }
    float mmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxSplits; ++c)
      if (c < nsplit) mmax = fmaxf(mmax, mc[c]);
    float lsum = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (mmax != -INFINITY) {
#pragma unroll
      for (int c = 0; c < kMaxSplits; ++c)
        if (c < nsplit) {
          const float f = exp2f(mc[c] - mmax);
          lsum += lc[c] * f;
          acc.x += vc[c].x * f;
          acc.y += vc[c].y * f;
          acc.z += vc[c].z * f;
          acc.w += vc[c].w * f;
        }
    }
    const float scale = mmax != -INFINITY ? p.kv_scale / lsum : 0.0f;
    uint2 packed;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed.x) : "f"(acc.y * scale), "f"(acc.x * scale));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed.y) : "f"(acc.w * scale), "f"(acc.z * scale));
    const int64_t head = static_cast<int64_t>(r) * p.heads + head0 + h;
    reinterpret_cast<uint2*>(p.out + head * 512)[d4] = packed;
    if (d4 == 0 && p.lse != nullptr)
      p.lse[head] = mmax != -INFINITY ? (mmax + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
  }
  cluster_sync();  // keep this CTA's shared memory alive until every reader is done
}

int g_max_splits_cache[64] = {0};

}  // namespace

void plan_mla_decode_cluster(DecodeParams& p) {
  int dev = 0;
  cudaGetDevice(&dev);
  int cap = kMaxSplits;
  if (dev >= 0 && dev < 64) {
    if (g_max_splits_cache[dev] == 0) {
      // Largest cluster (16, else 8) the device can schedule for this kernel.
      int best = 8;
      if (cudaFuncSetAttribute(mla_decode_cluster_kernel,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
          cudaFuncSetAttribute(mla_decode_cluster_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(Smem))) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = sizeof(Smem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, mla_decode_cluster_kernel, &cfg) ==
                cudaSuccess &&
            clusters > 0)
          best = 16;
      }
      cudaGetLastError();
      g_max_splits_cache[dev] = best;
    }
    cap = g_max_splits_cache[dev];
  }
  int n = (p.topk + 127) / 128;
  n = n < 1 ? 1 : (n > cap ? cap : n);
  int len = (p.topk + n - 1) / n;
  len = (len + kTok - 1) / kTok * kTok;
  p.splits = n;
  p.split_len = len;
}

cudaError_t launch_mla_decode_cluster(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(Smem);
  cudaError_t e = cudaFuncSetAttribute(mla_decode_cluster_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (p.splits > 8) {
    e = cudaFuncSetAttribute(mla_decode_cluster_kernel,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, (p.heads + kHG - 1) / kHG, p.rows.rows);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = dependent_launch_attr();
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mla_decode_cluster_kernel, p);
}

}  // namespace dsa
