// indexer_write.cu -- the indexer's write side for each row's new token: the
// k_norm LayerNorm (with a bias) of the row's wk projection, stored as bf16
// into the key arena at the row's device-side position.
//
// "glm5next_dsa/layer.rs", module header trap 2 (indexer.k_norm is an
// nn.LayerNorm with a bias: mean subtraction plus a bias term) and
// indexer_forward (k_raw = wk(hidden) lands in the cache row, LayerNorm in
// place, placement from a device-side position by dsa_indexer_store so that a
// captured graph does not freeze a host offset).
//
// One warp per row, index_dim / 32 elements per lane.  The statistics and the
// affine map are taken in double (at most 128 elements per row), and the
// result is rounded to bf16 once: round-to-odd from double to float, then
// round-to-nearest-even from float to bf16, which equals a direct
// round-to-nearest-even because float keeps 16 more bits than bf16 (Boldo and
// Melquiond, "Emulation of FMA and correctly rounded sums: proved algorithms
// using rounding to odd", IEEE Trans. Computers 57(4), 2008).
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ uint16_t bf16_rne_from_double(double v) {
  float f = __double2float_rz(v);
  if (static_cast<double>(f) != v && !isnan(v) && !isinf(f))
    f = __uint_as_float(__float_as_uint(f) | 1u);  // sticky bit: round to odd
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) indexer_write_kernel(const IndexerWriteParams p) {
  constexpr int kPer = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarps + warp;
  grid_dep_launch();
  if (r >= p.rows) return;  // whole warps only

  // The norm's weight and bias are weights (no kernel of a chain writes
  // them) and are read before the wait; the row metadata, k_raw and the gate
  // may come from kernels before, and the arena may still be read by one.
  double w[kPer], b[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    w[i] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(p.ln_w[lane * kPer + i]) << 16));
    b[i] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(p.ln_b[lane * kPer + i]) << 16));
  }
  grid_dep_wait();
  const int64_t pos = p.positions[r];
  const int64_t len = p.seq_lens[r];
  const int64_t base = p.idx_base[r];
  const int64_t t = base + pos;
  bool ok = true;
  if (pos + 1 != len) {
    if (lane == 0) record_error(p.err, DSA_DEVERR_POSITION, r);
    ok = false;
  } else if (base < 0 || t < 0 || t >= p.idx_tokens) {
    if (lane == 0) record_error(p.err, DSA_DEVERR_ARENA, r);
    ok = false;
  }

  if (!ok) return;
  double x[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i)
    x[i] = static_cast<double>(
        __uint_as_float(static_cast<uint32_t>(p.k_raw[static_cast<int64_t>(r) * D + lane * kPer + i]) << 16));
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) s += x[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  const double mu = s / D;
  double q = 0.0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) q += (x[i] - mu) * (x[i] - mu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xFFFFFFFFu, q, o);
  const double inv = 1.0 / sqrt(q / D + static_cast<double>(p.eps));
  uint16_t y[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) y[i] = bf16_rne_from_double((x[i] - mu) * inv * w[i] + b[i]);
  uint16_t* dst = p.idx_k + t * D + lane * kPer;
  if constexpr (kPer == 4) {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(static_cast<uint32_t>(y[0]) | (static_cast<uint32_t>(y[1]) << 16),
                   static_cast<uint32_t>(y[2]) | (static_cast<uint32_t>(y[3]) << 16));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = static_cast<uint32_t>(y[0]) | (static_cast<uint32_t>(y[1]) << 16);
  }
  if (p.gate != nullptr && lane == 0) p.idx_gate[t] = p.gate[r];
}

}  // namespace

cudaError_t launch_indexer_write(const IndexerWriteParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.rows + kWarps - 1) / kWarps), 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.dim == 64) return cudaLaunchKernelEx(&cfg, indexer_write_kernel<64>, p);
  return cudaLaunchKernelEx(&cfg, indexer_write_kernel<128>, p);
}

}  // namespace dsa
