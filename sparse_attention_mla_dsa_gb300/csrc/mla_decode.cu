// mla_decode.cu -- S3: absorbed NoPE MLA gather-attend of latent-space Q
// against the FP8 paged latent cache, over each row's selection only.
//
// "glm5next_dsa/layer.rs": module header trap 4 (Q arrives absorbed into the
// 512-wide latent space, so the kernel dots Q against the latent directly),
// attend_rows (one launch for all rows; each row has its own selection row,
// seq_len and block-table row; K and V are the same latent pool), decode_k
// (slot = block * block_size + pos % block_size).  Per row and head:
//     z_j = sm_scale * kv_scale * (Q . e4m3(latent_j)),  p = softmax(z)
//     out = kv_scale * sum_j p_j e4m3(latent_j),  lse = log sum_j exp(z_j)
//
// Split kernel: CTA = (split of 256 selection entries, 16 heads, row).  Each
// 32-token tile of selected latent rows is gathered with 16-byte cp.async
// (double-buffered), widened FP8 -> bf16 in shared memory (exact), and run
// through bf16 tensor-core MMAs for S = Q K^T and O += P V with an online
// softmax in between.  A combine kernel merges the splits in fixed split
// order.  The split count depends only on topk, so a row's result is the
// same bit for bit whatever other rows share the launch.
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 128;
constexpr int kHG = 16;        // heads per CTA
constexpr int kTok = 32;       // tokens per tile
constexpr int kSplit = 256;    // selection entries per split
constexpr int kRowB = 1040;    // bytes per bf16 row of 512 (+16 pad: conflict-free ldmatrix)
constexpr int kPRowB = 80;     // bytes per bf16 row of P (32 tokens + pad)

struct DecodeSmem {
  uint8_t q[kHG * kRowB];
  uint8_t kv[kTok * kRowB];
  uint8_t stage[2][kTok * 512];
  float s[kHG][kTok];
  uint8_t pmat[kHG * kPRowB];
  int64_t slot[kSplit];
  float m[kHG], l[kHG], alpha[kHG];
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

__global__ void __launch_bounds__(kThreads) mla_decode_split_kernel(const DecodeParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int split = blockIdx.x, hg = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = split * kSplit;
  const int nj = min(kSplit, p.topk - j0);
  const bool report = hg == 0;

  int len = p.rows.seq_lens[r];
  if (len < 0) {
    if (report && split == 0 && tid == 0) record_error(p.err, DSA_DEVERR_SEQ_LEN, r);
    len = 0;
  }
  const int32_t* bt = p.rows.block_table + static_cast<int64_t>(r) * p.rows.bt_stride;
  const int bs = p.rows.block_size;

  // Physical slot of every selected entry of this split (-1: padding / invalid).
  for (int i = tid; i < kSplit; i += kThreads) {
    int64_t slot = -1;
    if (i < nj) {
      const int idx = p.sel[static_cast<int64_t>(r) * p.topk + j0 + i];
      if (idx != -1) {
        if (idx < 0 || idx >= len) {
          if (report) record_error(p.err, DSA_DEVERR_SELECT, r);
        } else {
          const int blk = idx / bs;
          const int phys = blk < p.rows.max_blocks_per_seq ? bt[blk] : -1;
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
  // Q tile: heads hg*16 .. +15 of row r.
  const uint16_t* qsrc = p.q + (static_cast<int64_t>(r) * p.heads + hg * kHG) * 512;
  for (int c = tid; c < kHG * 64; c += kThreads) {
    const int h = c >> 6, k = c & 63;
    cp_async16(sm.q + h * kRowB + k * 16, qsrc + h * 512 + k * 8, 16);
  }
  cp_async_commit();
  if (tid < kHG) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.0f;
  }
  __syncthreads();

  const int ntiles = (nj + kTok - 1) / kTok;
  auto issue_tile = [&](int tile, int buf) {
    for (int c = tid; c < kTok * 32; c += kThreads) {
      const int tok = c >> 5, k = c & 31;
      const int i = tile * kTok + tok;
      const int64_t slot = i < nj ? sm.slot[i] : -1;
      const uint8_t* src = slot >= 0 ? p.pool + slot * 512 + k * 16 : p.pool;
      cp_async16(&sm.stage[buf][tok * 512 + k * 16], src, slot >= 0 ? 16u : 0u);
    }
    cp_async_commit();
  };
  if (ntiles > 0) issue_tile(0, 0);

  float o[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.0f;
  const float scale_log2 = p.sm_scale * p.kv_scale * 1.4426950408889634f;
  const int g = lane >> 2, t2 = (lane & 3) * 2;

  for (int it = 0; it < ntiles; ++it) {
    if (it + 1 < ntiles) {
      issue_tile(it + 1, (it + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // FP8 -> bf16 (exact) into the padded latent tile.
    const uint8_t* st = sm.stage[it & 1];
    for (int c = tid; c < kTok * 32; c += kThreads) {
      const int tok = c >> 5, k = c & 31;
      const uint4 raw = *reinterpret_cast<const uint4*>(st + tok * 512 + k * 16);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t cv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cv[2 * i] = e4m3x2_to_bf16x2(static_cast<uint16_t>(w[i] & 0xFFFFu));
        cv[2 * i + 1] = e4m3x2_to_bf16x2(static_cast<uint16_t>(w[i] >> 16));
      }
      uint4* dst = reinterpret_cast<uint4*>(sm.kv + tok * kRowB + k * 32);
      dst[0] = make_uint4(cv[0], cv[1], cv[2], cv[3]);
      dst[1] = make_uint4(cv[4], cv[5], cv[6], cv[7]);
    }
    __syncthreads();

    // S = Q K^T: warp w takes tokens 8w .. 8w+7 against all 16 heads.
    {
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      const uint32_t a_addr =
          smem_u32(sm.q) + ((lane & 7) + ((lane >> 3) & 1) * 8) * kRowB + (lane >> 4) * 16;
      const uint32_t b_addr =
          smem_u32(sm.kv) + (warp * 8 + (lane & 7)) * kRowB + ((lane >> 3) & 1) * 16;
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1;
        ldsm_x4(a_addr + kk * 32, a0, a1, a2, a3);
        ldsm_x2(b_addr + kk * 32, b0, b1);
        mma_bf16_16816(acc, a0, a1, a2, a3, b0, b1);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = g + (e >> 1) * 8, tok = warp * 8 + t2 + (e & 1);
        const int i = it * kTok + tok;
        const bool valid = i < nj && sm.slot[i] >= 0;
        sm.s[h][tok] = valid ? acc[e] * scale_log2 : -INFINITY;
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
      prow[0] = pack_bf16x2(pv[0], pv[1]);
      prow[1] = pack_bf16x2(pv[2], pv[3]);
      if ((tid & 7) == 0) {
        sm.l[h] = sm.l[h] * alpha + psum;
        sm.m[h] = m_new;
        sm.alpha[h] = alpha;
      }
    }
    __syncthreads();

    // O = alpha * O + P V: warp w owns latent dims 128w .. 128w+127.
    {
      const float al0 = sm.alpha[g], al1 = sm.alpha[g + 8];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] *= al0;
        o[nt][1] *= al0;
        o[nt][2] *= al1;
        o[nt][3] *= al1;
      }
      const uint32_t pbase = smem_u32(sm.pmat), kvbase = smem_u32(sm.kv);
#pragma unroll
      for (int ks = 0; ks < kTok / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(pbase + ((lane & 7) + ((lane >> 3) & 1) * 8) * kPRowB + ks * 32 + (lane >> 4) * 16,
                a0, a1, a2, a3);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          const int d0 = warp * 128 + np * 16;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(kvbase + (ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kRowB +
                            (d0 + (lane >> 4) * 8) * 2,
                        b0, b1, b2, b3);
          mma_bf16_16816(o[2 * np], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
  }

  // Unnormalised partial of this split.
  const int64_t part = (static_cast<int64_t>(r) * p.splits + split) * p.heads + hg * kHG;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int d = warp * 128 + nt * 8 + t2;
    *reinterpret_cast<float2*>(p.part_o + (part + g) * 512 + d) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(p.part_o + (part + g + 8) * 512 + d) =
        make_float2(o[nt][2], o[nt][3]);
  }
  if (tid < kHG)
    *reinterpret_cast<float2*>(p.part_ml + (part + tid) * 2) = make_float2(sm.m[tid], sm.l[tid]);
}

// Merge the splits of one (row, head) in fixed split order.
__global__ void __launch_bounds__(kThreads) mla_decode_combine_kernel(const DecodeParams p) {
  const int h = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  const int64_t base = static_cast<int64_t>(r) * p.splits * p.heads + h;
  float mmax = -INFINITY;
  for (int s = 0; s < p.splits; ++s) mmax = fmaxf(mmax, p.part_ml[(base + s * p.heads) * 2]);
  float lsum = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (mmax != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const int64_t ps = base + static_cast<int64_t>(s) * p.heads;
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + ps * 2);
      const float f = exp2f(ml.x - mmax);
      lsum += ml.y * f;
      const float4 v = reinterpret_cast<const float4*>(p.part_o + ps * 512)[tid];
      acc.x += v.x * f;
      acc.y += v.y * f;
      acc.z += v.z * f;
      acc.w += v.w * f;
    }
  }
  const float scale = mmax != -INFINITY ? p.kv_scale / lsum : 0.0f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * scale, acc.y * scale);
  packed.y = pack_bf16x2(acc.z * scale, acc.w * scale);
  reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(r) * p.heads + h) * 512)[tid] = packed;
  if (tid == 0 && p.lse != nullptr)
    p.lse[static_cast<int64_t>(r) * p.heads + h] =
        mmax != -INFINITY ? (mmax + log2f(lsum)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int32_t decode_splits(int32_t topk) { return (topk + kSplit - 1) / kSplit; }

size_t decode_workspace_bytes(int32_t rows, int32_t heads, int32_t topk) {
  const size_t n = static_cast<size_t>(rows) * decode_splits(topk) * heads;
  const size_t o_bytes = (n * 512 * sizeof(float) + 255) & ~static_cast<size_t>(255);
  return o_bytes + n * 2 * sizeof(float);
}

cudaError_t launch_mla_decode(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = sizeof(DecodeSmem);
  cudaError_t e = cudaFuncSetAttribute(mla_decode_split_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.splits, p.heads / kHG, p.rows.rows);
  mla_decode_split_kernel<<<grid, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mla_decode_combine_kernel<<<dim3(p.heads, p.rows.rows), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
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
// on the decode path.  This entry point runs the two-kernel split + combine
// form above (no thread-block clusters) with its split partials in this
// file-scope device array instead of a caller-provided workspace.  The array
// is DSA_NOALLOC_SCRATCH_BYTES long and every GPU that loads the library keeps
// it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[64] = {};
}  // namespace

extern "C" size_t dsa_noalloc_scratch_bytes(int32_t rows, int32_t heads, int32_t topk) {
  if (rows < 1 || heads < 1 || topk < 1) return 0;
  return dsa::decode_workspace_bytes(rows, heads, topk);
}

extern "C" dsa_status dsa_mla_decode_fp8_noalloc(const dsa_rows* rows, const uint16_t* q,
                                                 const uint8_t* pool, int64_t nslots,
                                                 const int32_t* sel, int32_t topk, int32_t heads,
                                                 int32_t latent_dim, float kv_scale,
                                                 float sm_scale, uint16_t* out,
                                                 float* lse_or_null, void* stream) {
  if (rows == nullptr || rows->rows < 1 || rows->rows > 65535 || rows->seq_lens == nullptr ||
      rows->block_table == nullptr || rows->block_size < 1 || rows->max_blocks_per_seq < 1 ||
      rows->bt_stride < 0 || (rows->bt_stride != 0 && rows->bt_stride < rows->max_blocks_per_seq))
    return DSA_ERR_INVALID_ARG;
  if (q == nullptr || pool == nullptr || sel == nullptr || out == nullptr || nslots < 1)
    return DSA_ERR_INVALID_ARG;
  if (latent_dim != DSA_LATENT_DIM) return DSA_ERR_UNSUPPORTED;
  if (heads < 16 || heads % 16 != 0 || heads > 4096) return DSA_ERR_UNSUPPORTED;
  if (topk < 1 || topk > 65536) return DSA_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(pool) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 7))
    return DSA_ERR_INVALID_ARG;
  if (dsa::decode_workspace_bytes(rows->rows, heads, topk) > DSA_NOALLOC_SCRATCH_BYTES)
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
  int* err = dsa::device_error_word();
  if (err == nullptr) return DSA_ERR_CUDA;
  dsa::DecodeParams p{};
  p.rows = *rows;
  p.q = q;
  p.pool = pool;
  p.nslots = nslots;
  p.sel = sel;
  p.out = out;
  p.lse = lse_or_null;
  p.topk = topk;
  p.heads = heads;
  p.splits = dsa::decode_splits(topk);
  const size_t n = static_cast<size_t>(rows->rows) * p.splits * heads;
  p.part_o = static_cast<float*>(scratch);
  p.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) +
                                       ((n * 512 * sizeof(float) + 255) & ~static_cast<size_t>(255)));
  p.err = err;
  p.kv_scale = kv_scale;
  p.sm_scale = sm_scale;
  return dsa::launch_mla_decode(p, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}
