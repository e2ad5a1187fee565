// latent_write.cu -- S0: vanilla RMSNorm + FP8 E4M3 quantisation + paged
// slot write of each row's new latent.
//
// "glm5next_dsa/layer.rs", module header trap 1 (GLM's norm is x*rms*w, the
// +1 variant is a different kernel) and decode_k "kv path: latent -> FP8 ->
// paged slot" (the write receives eps and 1/kv_scale as f32 and a slot
// block*block_size + pos%block_size); "Struct Glm5NextDsaLayer", kv_scale.
//
// One CTA of 128 threads per row, 4 latent elements per thread.  The norm is
// taken in double (512 elements per row: the FP64 units are nowhere near a
// bound here), so the only rounding that matters is the final one to E4M3,
// done by encode_e4m3_rne below from the format's definition.
#include "dsa_device.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 128;

// Round-to-nearest-even of a double to OCP E4M3 with saturation to +-448.
// Normal range: |v| = 2^e * q/8 with q in [8,16); subnormal: |v| = q * 2^-9.
__device__ __forceinline__ uint8_t encode_e4m3_rne(double v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  const double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  if (a < 0.015625) {  // below 2^-6: subnormal spacing 2^-9
    const int q = static_cast<int>(rint(a * 512.0));  // 0..8; 8 is the first normal code
    return sign | static_cast<uint8_t>(q);
  }
  int e = ilogb(a);                                     // 2^e <= a < 2^(e+1), e in [-6, 8]
  int q = static_cast<int>(rint(scalbn(a, 3 - e)));     // 8..16
  if (q == 16) {
    q = 8;
    ++e;
  }
  return sign | static_cast<uint8_t>(((e + 7) << 3) | (q - 8));
}

__global__ void __launch_bounds__(kThreads) latent_write_kernel(LatentWriteParams p) {
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  __shared__ double warp_sum[kThreads / 32];
  __shared__ int skip;
  grid_dep_launch();
  // Every input may be the output of the kernel before (kv_a from a
  // projection, metadata written on the device), and the previous
  // gather-attend may still read the pool: nothing is read or written before
  // the wait.
  grid_dep_wait();

  if (tid == 0) {
    int bad = 0;
    const int64_t slot = p.rows.slots[r];
    if (slot < 0 || slot >= p.nslots) {
      record_error(p.err, DSA_DEVERR_SLOT, r);
      bad = 1;
    } else if (p.rows.positions != nullptr) {
      // The two encodings of the row's place must agree: position = seq_len-1
      // and slot = table[pos / block_size] * block_size + pos % block_size.
      const int64_t pos = p.rows.positions[r];
      const int64_t len = p.rows.seq_lens[r];
      const int64_t blk = pos / p.rows.block_size;
      const int32_t* bt = p.rows.block_table + static_cast<int64_t>(r) * p.rows.bt_stride;
      if (pos < 0 || pos + 1 != len || blk >= p.rows.max_blocks_per_seq ||
          static_cast<int64_t>(bt[blk]) * p.rows.block_size + pos % p.rows.block_size != slot) {
        record_error(p.err, DSA_DEVERR_POSITION, r);
        bad = 1;
      }
    }
    skip = bad;
  }

  // 4 bf16 inputs per thread.
  const uint2 xin = reinterpret_cast<const uint2*>(p.kv_a + static_cast<int64_t>(r) * 512)[tid];
  const uint2 win = reinterpret_cast<const uint2*>(p.norm_w)[tid];
  double x[4], w[4];
  const uint32_t xs[2] = {xin.x, xin.y}, ws[2] = {win.x, win.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    x[2 * i] = static_cast<double>(__uint_as_float(xs[i] << 16));
    x[2 * i + 1] = static_cast<double>(__uint_as_float(xs[i] & 0xFFFF0000u));
    w[2 * i] = static_cast<double>(__uint_as_float(ws[i] << 16));
    w[2 * i + 1] = static_cast<double>(__uint_as_float(ws[i] & 0xFFFF0000u));
  }
  double ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((tid & 31) == 0) warp_sum[tid >> 5] = ss;
  __syncthreads();
  if (skip) return;
  const double total = (warp_sum[0] + warp_sum[1]) + (warp_sum[2] + warp_sum[3]);
  const double rms = 1.0 / sqrt(total / 512.0 + static_cast<double>(p.eps));
  const double inv = static_cast<double>(p.inv_scale);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const double y = x[i] * rms * w[i];
    packed |= static_cast<uint32_t>(encode_e4m3_rne(y * inv)) << (8 * i);
  }
  const int64_t slot = p.rows.slots[r];
  reinterpret_cast<uint32_t*>(p.pool + slot * 512)[tid] = packed;
}

}  // namespace

cudaError_t launch_latent_write(const LatentWriteParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows.rows, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {dependent_launch_attr()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, latent_write_kernel, p);
}

}  // namespace dsa
