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
// The lockstep of the indexer cache with the KV cache (decode_k: the
// indexer's length must equal the sequence length before the step; a longer
// cache is the leftover of a rejected verify and is rewound, a shorter one
// means rows were never written and is a hard error): with a per-sequence
// counter of written rows, the rows of a sequence (consecutive positions
// p0, p0+1, ... of one call) are written only when the counter is at least
// p0, and the counter becomes p0 + rows afterwards; a counter below p0 is
// recorded as DSA_DEVERR_BEHIND and nothing of that sequence is written.
//
// One warp per row, index_dim / 32 elements per lane; with the counter, one
// CTA per sequence (a warp per row of it).  The statistics and the
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
__device__ __forceinline__ void write_row(const IndexerWriteParams& p, int r, int lane,
                                          const double (&w)[D / 32], const double (&b)[D / 32]) {
  constexpr int kPer = D / 32;
  const int64_t pos = p.positions[r];
  const int64_t len = p.seq_lens[r];
  const int64_t base = p.idx_base[r];
  const int64_t t = base + pos;
  if (pos + 1 != len) {
    if (lane == 0) record_error(p.err, DSA_DEVERR_POSITION, r);
    return;
  }
  if (base < 0 || t < 0 || t >= p.idx_tokens) {
    if (lane == 0) record_error(p.err, DSA_DEVERR_ARENA, r);
    return;
  }
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

template <int D>
__device__ __forceinline__ void load_norm(const IndexerWriteParams& p, int lane, double (&w)[D / 32],
                                          double (&b)[D / 32]) {
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    w[i] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(p.ln_w[lane * (D / 32) + i]) << 16));
    b[i] = static_cast<double>(__uint_as_float(static_cast<uint32_t>(p.ln_b[lane * (D / 32) + i]) << 16));
  }
}

// Without the counter: one warp per row, four rows per CTA.
template <int D>
__global__ void __launch_bounds__(kWarps * 32) indexer_write_kernel(const IndexerWriteParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarps + warp;
  grid_dep_launch();
  if (r >= p.rows) return;  // whole warps only
  // The norm's weight and bias are weights (no kernel of a chain writes
  // them) and are read before the wait; the row metadata, k_raw and the gate
  // may come from kernels before, and the arena may still be read by one.
  double w[D / 32], b[D / 32];
  load_norm<D>(p, lane, w, b);
  grid_dep_wait();
  write_row<D>(p, r, lane, w, b);
}

// With the counter: one CTA per sequence, a warp per row of it.
template <int D>
__global__ void __launch_bounds__(32 * 32) indexer_write_lockstep_kernel(const IndexerWriteParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = blockIdx.x, r0 = seq * p.rows_per_seq;
  __shared__ int write_ok;
  grid_dep_launch();
  double w[D / 32], b[D / 32];
  load_norm<D>(p, lane, w, b);
  grid_dep_wait();
  if (threadIdx.x == 0) {
    const int64_t written = p.idx_written[seq];
    const int64_t p0 = p.positions[r0];
    // behind: rows [written, p0) of this sequence were never written
    write_ok = written >= p0 ? 1 : 0;
    if (!write_ok) record_error(p.err, DSA_DEVERR_BEHIND, r0);
  }
  __syncthreads();
  if (write_ok && warp < p.rows_per_seq) {
    const int r = r0 + warp;
    if (static_cast<int64_t>(p.positions[r]) != static_cast<int64_t>(p.positions[r0]) + warp) {
      if (lane == 0) record_error(p.err, DSA_DEVERR_POSITION, r);
    } else {
      write_row<D>(p, r, lane, w, b);
    }
  }
  __syncthreads();
  // ahead (a rejected verify's rows) or level: the sequence now holds
  // exactly the rows up to its last new position
  if (threadIdx.x == 0 && write_ok)
    p.idx_written[seq] = static_cast<int32_t>(static_cast<int64_t>(p.positions[r0]) + p.rows_per_seq);
}

}  // namespace

cudaError_t launch_indexer_write(const IndexerWriteParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.idx_written != nullptr) {
    cfg.gridDim = dim3(static_cast<unsigned>(p.rows / p.rows_per_seq), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * p.rows_per_seq), 1, 1);
    if (p.dim == 64) return cudaLaunchKernelEx(&cfg, indexer_write_lockstep_kernel<64>, p);
    return cudaLaunchKernelEx(&cfg, indexer_write_lockstep_kernel<128>, p);
  }
  cfg.gridDim = dim3(static_cast<unsigned>((p.rows + kWarps - 1) / kWarps), 1, 1);
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  if (p.dim == 64) return cudaLaunchKernelEx(&cfg, indexer_write_kernel<64>, p);
  return cudaLaunchKernelEx(&cfg, indexer_write_kernel<128>, p);
}

}  // namespace dsa
