// Standalone dequantisation to fp32 [K, N] and the one-time repack into the
// tensor-core operand layout.
#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

// ----------------------------------------------------------------------------------
// Dequant: out[k * N + n] = (code - zp) * scale, rounded once to fp32, as the
// matmul_nbits_dequant_f32 kernel of matmul_nbits.rs writes it.  HBM write-bound
// (4 bytes written per half byte read), so the CTA transposes a 64 x 64 tile through
// shared memory: reads are whole 8-byte pieces of weight rows, writes are 64-float
// runs of output rows.
// ----------------------------------------------------------------------------------
struct DequantArgs {
  const uint8_t* packed;
  const void* scales;
  const uint8_t* zp;
  int scales_f16;
  float* out;
  int K, N, G, zrb, bs;
};

__global__ void __launch_bounds__(256) dequant_kernel(const DequantArgs p) {
  __shared__ float tile[64][65];
  const int tid = threadIdx.x;
  const int ntn = (p.N + 63) >> 6;
  const int n_base = (int)(blockIdx.x % ntn) * 64, k_base = (int)(blockIdx.x / ntn) * 64;
  pdl_launch_dependents();
  pdl_wait();
  {
    const int c = tid >> 2, q = tid & 3;  // column in tile, 16-element piece
    const int n = n_base + c, k = k_base + 16 * q;
    if (n < p.N && k < p.K) {
      const uint2 wv = *reinterpret_cast<const uint2*>(p.packed + (long long)n * (p.K >> 1) + (k >> 1));
      const int g = k / p.bs;
      int z = 8;
      if (p.zp) {
        const uint32_t b = p.zp[(long long)n * p.zrb + (g >> 1)];
        z = (g & 1) ? (int)(b >> 4) : (int)(b & 15u);
      }
      const long long si = (long long)n * p.G + g;
      const float s = p.scales_f16 ? __half2float(reinterpret_cast<const __half*>(p.scales)[si])
                                   : reinterpret_cast<const float*>(p.scales)[si];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        tile[16 * q + i][c] = __fmul_rn((float)((int)((wv.x >> (4 * i)) & 15u) - z), s);
        tile[16 * q + 8 + i][c] = __fmul_rn((float)((int)((wv.y >> (4 * i)) & 15u) - z), s);
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < 64 * 64; e += 256) {
    const int kk = e >> 6, nn = e & 63;
    const int k = k_base + kk, n = n_base + nn;
    if (k < p.K && n < p.N) p.out[(long long)k * p.N + n] = tile[kk][nn];
  }
}

// ----------------------------------------------------------------------------------
// Repack.  Output chunk idx (16 bytes) is block idx / 256 (tile t, k-block b), part
// q = (idx / 128) % 2, row r = idx % 128, so the output is written sequentially.  Each
// 32-bit word keeps its eight k but moves the even-k nibbles to the low half-word and the
// odd-k nibbles to the high half-word: word nibble p then holds k offset 2(p%4) + p/4.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t split_even_odd_nibbles(uint32_t w) {
  uint32_t r = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    r |= ((w >> (8 * p)) & 15u) << (4 * p);
    r |= ((w >> (8 * p + 4)) & 15u) << (16 + 4 * p);
  }
  return r;
}

__global__ void __launch_bounds__(256) repack_kernel(const uint8_t* __restrict__ packed,
                                                     uint8_t* __restrict__ out, int K, int N,
                                                     int kblocks, long long chunks) {
  pdl_launch_dependents();
  pdl_wait();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= chunks) return;
  const long long blk = idx >> 8;
  const int within = (int)(idx & 255);
  const int q = within >> 7, r = within & 127;
  const long long t = blk / kblocks;
  const int b = (int)(blk - t * kblocks);
  const long long n = t * 128 + r;
  const int k0 = b * 64 + q * 32;
  uint32_t w[4] = {0, 0, 0, 0};
  if (n < N) {
    const uint8_t* row = packed + n * (long long)(K >> 1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + 8 * j;
      if (k < K) w[j] = split_even_odd_nibbles(*reinterpret_cast<const uint32_t*>(row + (k >> 1)));
    }
  }
  *reinterpret_cast<uint4*>(out + idx * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

cudaError_t launch_dequant(LaunchCtx& ctx, const QWeight& w, int K, int N, int bs, float* out) {
  DequantArgs a = {};
  a.packed = w.packed;
  a.scales = w.scales;
  a.zp = w.zp;
  a.scales_f16 = w.scales_f16;
  a.out = out;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.bs = bs;
  const long long tiles = (long long)((N + 63) / 64) * ((K + 63) / 64);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ctx.variant = "dequant_f32_tile64";
  return launch_kernel(ctx, dequant_kernel, dim3((unsigned)tiles), dim3(256), 0, a);
}

cudaError_t launch_repack(LaunchCtx& ctx, const uint8_t* packed, int K, int N, uint8_t* out) {
  const int kblocks = (K + 63) / 64;
  const long long ntiles = (N + 127) / 128;
  const long long chunks = ntiles * kblocks * 256;
  const unsigned grid = (unsigned)((chunks + 255) / 256);
  ctx.variant = "repack_tc_tiles";
  return launch_kernel(ctx, repack_kernel, dim3(grid), dim3(256), 0, packed, out, K, N, kblocks,
                       chunks);
}

}  // namespace mnb
