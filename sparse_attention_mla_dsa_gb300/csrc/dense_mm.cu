// dense_mm.cu -- batched projection for the K-token verify: one sweep of a
// BF16 weight serves up to 16 activation rows.
//
// "glm5next_dsa/layer.rs", the gemm helper (C[M, N] = A[M, K] @ B[N, K]^T)
// and the notes on decode_k / dense_gemv_bf16_batchm: the K rows of one
// sequence sweep each projection weight once, and each row's result must be
// bit-identical to a single-row call.
//
// Mapping onto the tensor core ("swap AB": weight rows are M):
//   A = 128 weight rows x 64 of K (bf16, K-major, TMA with 128-byte swizzle)
//   B = 16 activation rows x 64 of K; rows >= M lie past the tensor map and
//       arrive as zeros, so the instruction is the same for every M
//   D = 128 x 16 FP32 accumulators in TMEM (lane = weight row, column = row m)
// Each output column is a function of its own activation row and the weight
// only, and the K split of a launch depends on (N, K) and the SM count only:
// a row's result does not depend on M or on what the other rows hold.
//
// CTA roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues the
// MMAs (one thread), warps 2-5 are the epilogue (one TMEM lane quarter each).
// A CTA handles one 128-row weight tile over one contiguous range of K; with
// more than one range per tile the FP32 partials go to the workspace and a
// second kernel adds them in range order.
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kTileN = 128;                          // weight rows per tile (MMA M)
constexpr int kRowsPad = 16;                         // activation rows (MMA N)
constexpr int kBlockK = 64;                          // K per stage: one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr int kStages = 6;
constexpr uint32_t kWBytes = kTileN * kBlockK * 2;   // 16 KB weight tile
constexpr uint32_t kABytes = kRowsPad * kBlockK * 2; // 2 KB activation tile
constexpr uint32_t kStageBytes = kWBytes + kABytes;
constexpr uint32_t kTmemCols = 32;                   // 16 used; 32 is the allocation minimum
static_assert(kStageBytes % 1024 == 0, "stage bases must stay 1024-byte aligned");

struct __align__(8) MmCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kSmemBytes = kStages * kStageBytes + sizeof(MmCtl) + 1024;  // + alignment slack

__device__ __forceinline__ void set_abort(MmCtl* c, int* err, int tile) {
  record_error(err, DSA_DEVERR_TIMEOUT, tile);
  *reinterpret_cast<volatile int*>(&c->abort_flag) = 1;
}
__device__ __forceinline__ bool aborted(MmCtl* c) {
  return *reinterpret_cast<volatile int*>(&c->abort_flag) != 0;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__global__ void __launch_bounds__(kThreads, 1)
    dense_mm_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
                    const DenseMmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  MmCtl* ctl = reinterpret_cast<MmCtl*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, tile = blockIdx.y;
  const int kb_begin = split * p.kb_per_split;
  const int nkb = min(p.kb_per_split, p.kblocks - kb_begin);  // >= 1 by the plan
  const int n0 = tile * kTileN;
  grid_dep_launch();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->tfull, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&wmap);
    tma_prefetch_map(&amap);
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // Weights stream through once (evict first); the activation tiles are
      // read by every weight tile of the launch (keep them).
      const uint64_t w_policy = l2_policy_evict_first();
      const uint64_t a_policy = l2_policy_evict_normal();
      // The weight is an input no kernel writes: the first stages' weight
      // tiles go out before the dependency wait (overlapping the tail of the
      // kernel before), their activation tiles after it, on the same barrier.
      const int early = min(nkb, kStages);
      for (int i = 0; i < early; ++i) {
        mbar_arrive_expect_tx(&ctl->full[i], kStageBytes);
        tma_load_2d(smem + i * kStageBytes, &wmap, &ctl->full[i], (kb_begin + i) * kBlockK, n0,
                    w_policy);
      }
      grid_dep_wait();  // the activations may come from the kernel before
      for (int i = 0; i < early; ++i)
        tma_load_2d(smem + i * kStageBytes + kWBytes, &amap, &ctl->full[i], (kb_begin + i) * kBlockK,
                    0, a_policy);
      int issued = early;
      for (; issued < nkb; ++issued) {
        if (aborted(ctl)) break;
        const int s = issued % kStages;
        if (issued >= kStages &&
            !mbar_wait(&ctl->empty[s], ((issued / kStages) - 1) & 1, p.wait_ns)) {
          set_abort(ctl, p.err, tile);
          break;
        }
        uint8_t* dst = smem + s * kStageBytes;
        const int32_t x = (kb_begin + issued) * kBlockK;
        mbar_arrive_expect_tx(&ctl->full[s], kStageBytes);
        tma_load_2d(dst, &wmap, &ctl->full[s], x, n0, w_policy);
        tma_load_2d(dst + kWBytes, &amap, &ctl->full[s], x, 0, a_policy);
      }
      // Never leave with a copy in flight: wait (bounded) for the last loads.
      for (int i = max(0, issued - kStages); i < issued; ++i)
        mbar_wait(&ctl->full[i % kStages], (i / kStages) & 1, kDrainWaitNs);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kTileN, kRowsPad);
      const uint32_t base = smem_u32(smem);
      int done = 0;
      for (; done < nkb; ++done) {
        if (aborted(ctl)) break;
        const int s = done % kStages;
        if (!mbar_wait(&ctl->full[s], (done / kStages) & 1, p.wait_ns)) {
          set_abort(ctl, p.err, tile);
          break;
        }
        tc_fence_after();
        const uint32_t w_addr = base + s * kStageBytes;
        const uint32_t a_addr = w_addr + kWBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockK / 16; ++kk)
          umma_bf16(tmem, umma_desc_sw128_kmajor(w_addr + kk * 32),
                    umma_desc_sw128_kmajor(a_addr + kk * 32), idesc, (done | kk) != 0);
        umma_commit(&ctl->empty[s]);
      }
      // The epilogue always gets its signal; after an abort it writes nothing.
      umma_commit(&ctl->tfull);
      umma_commit(&ctl->drain);
      mbar_wait(&ctl->drain, 0, kDrainWaitNs);
    }
  } else {
    // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. those weight rows.
    const int quarter = warp & 3;
    const int n = n0 + quarter * 32 + lane;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&ctl->tfull, 0, p.wait_ns) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok && lane == 0) set_abort(ctl, p.err, tile);
    const bool write = ok && !__shfl_sync(0xFFFFFFFFu, aborted(ctl) ? 1 : 0, 0);
    tc_fence_after();
    float v[16];
    if (ok) {  // (uniform over the warp: tcgen05.ld is warp-collective)
      tmem_load16(tmem + (static_cast<uint32_t>(quarter * 32) << 16), v);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    }
    grid_dep_wait();  // the kernel before may still read the output
    if (write && n < p.n) {
      if (p.splits > 1) {
        float* dst = p.part + static_cast<int64_t>(split) * p.m * p.n + n;
#pragma unroll
        for (int m = 0; m < kRowsPad; ++m)
          if (m < p.m) dst[static_cast<int64_t>(m) * p.n] = v[m];
      } else if (p.c_fp32) {
        float* dst = static_cast<float*>(p.c) + n;
#pragma unroll
        for (int m = 0; m < kRowsPad; ++m)
          if (m < p.m) dst[static_cast<int64_t>(m) * p.n] = v[m];
      } else {
        uint16_t* dst = static_cast<uint16_t*>(p.c) + n;
#pragma unroll
        for (int m = 0; m < kRowsPad; ++m)
          if (m < p.m) dst[static_cast<int64_t>(m) * p.n] = __bfloat16_as_ushort(__float2bfloat16_rn(v[m]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Sum of the K ranges of each output, in range order, then the output type.
__global__ void __launch_bounds__(256) dense_mm_reduce_kernel(const DenseMmParams p) {
  grid_dep_wait();  // the partials come from the kernel before
  grid_dep_launch();
  const int64_t total = static_cast<int64_t>(p.m) * p.n;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  // Eight partials in flight per round trip, added in range order.
  float s = 0.0f;
  for (int r0 = 0; r0 < p.splits; r0 += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = r0 + u < p.splits ? p.part[(r0 + u) * total + i] : 0.0f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (r0 + u < p.splits) s = (r0 + u == 0) ? v[u] : s + v[u];
  }
  if (p.c_fp32)
    static_cast<float*>(p.c)[i] = s;
  else
    static_cast<uint16_t*>(p.c)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(s));
}

}  // namespace

void plan_dense_mm(DenseMmParams& p, int num_sms) {
  p.tiles = (p.n + kTileN - 1) / kTileN;
  p.kblocks = (p.k + kBlockK - 1) / kBlockK;
  // Split K only when the weight tiles alone leave SMs idle, and keep at
  // least four K blocks (64 KB of weight) per CTA.
  int splits = 1;
  if (p.tiles < num_sms) splits = (num_sms + p.tiles - 1) / p.tiles;
  const int max_splits = p.kblocks / 4 > 1 ? p.kblocks / 4 : 1;
  splits = splits < max_splits ? splits : max_splits;
  p.kb_per_split = (p.kblocks + splits - 1) / splits;
  p.splits = (p.kblocks + p.kb_per_split - 1) / p.kb_per_split;  // no empty range
}

size_t dense_mm_workspace_bytes(int32_t n, int32_t k, int num_sms) {
  DenseMmParams p{};
  p.n = n;
  p.k = k;
  plan_dense_mm(p, num_sms);
  if (p.splits <= 1) return 0;
  return static_cast<size_t>(p.splits) * kRowsPad * static_cast<size_t>(n) * sizeof(float);
}

cudaError_t launch_dense_mm(const DenseMmParams& p, const CUtensorMap& wmap,
                            const CUtensorMap& amap, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(dense_mm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  if (p.tiles > 65535 || p.splits > 65535) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.splits), static_cast<unsigned>(p.tiles), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, dense_mm_kernel, wmap, amap, p);
  if (e != cudaSuccess || p.splits <= 1) return e;
  const int64_t total = static_cast<int64_t>(p.m) * p.n;
  cudaLaunchConfig_t rcfg = {};
  rcfg.gridDim = dim3(static_cast<unsigned>((total + 255) / 256), 1, 1);
  rcfg.blockDim = dim3(256, 1, 1);
  rcfg.stream = stream;
  rcfg.attrs = attr;
  rcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&rcfg, dense_mm_reduce_kernel, p);
}

}  // namespace dsa
