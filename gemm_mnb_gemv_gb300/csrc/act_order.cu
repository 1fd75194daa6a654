// Act-order (g_idx) weights: dequantisation with a group index per k, the one-time
// preparation of an equivalent block-layout weight, and the per-call activation gather.
//
// The pages apply g_idx inside a dequantise-then-GEMM path (matmul_nbits.rs,
// matmul_nbits_dequant_f32: the scale and zero point of column k come from group
// g_idx[k], the code from block k / bs), with a device-to-host copy that checks every
// entry on each call.  Here the check and the reordering happen once, when the weight
// is prepared: k is sorted by group (ascending k inside a group), each group's run is
// padded to whole blocks, and the codes are gathered into that order.  The result is a
// plain MatMulNBits weight of K' >= K columns, so every call runs the block kernels
// unchanged on the gathered activation A'[m, k'] = A[m, perm[k']] (0 at a padding slot).
#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

__device__ __forceinline__ uint32_t nibble_at(const uint8_t* row, int k) {
  const uint32_t b = row[k >> 1];
  return (k & 1) ? (b >> 4) : (b & 15u);
}

// ----------------------------------------------------------------------------------
// Dequant with g_idx: out[k * N + n] = (code[n, k] - zp[n, g]) * scale[n, g] with
// g = g_idx[k], rounded once to fp32; 0 where g is outside 0..G-1 (which also sets
// kStatusBadIndex).  Same 64 x 64 shared-memory transpose as the plain dequant.
// ----------------------------------------------------------------------------------
struct DequantGidxArgs {
  const uint8_t* packed;
  const void* scales;
  const uint8_t* zp;
  const int32_t* gidx;
  int scales_f16;
  float* out;
  int K, N, G, zrb;
  uint32_t* status;
};

__global__ void __launch_bounds__(256) dequant_gidx_kernel(const DequantGidxArgs p) {
  __shared__ float tile[64][65];
  const int tid = threadIdx.x;
  const int ntn = (p.N + 63) >> 6;
  const int n_base = (int)(blockIdx.x % ntn) * 64, k_base = (int)(blockIdx.x / ntn) * 64;
  pdl_launch_dependents();
  pdl_wait();
  {
    const int c = tid >> 2, q = tid & 3;
    const int n = n_base + c, k = k_base + 16 * q;
    if (n < p.N && k < p.K) {  // K % 16 == 0, so k + 15 < K
      const uint2 wv = *reinterpret_cast<const uint2*>(p.packed + (long long)n * (p.K >> 1) + (k >> 1));
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int g = p.gidx[k + i];
        float v = 0.0f;
        if (g >= 0 && g < p.G) {
          int z = 8;
          if (p.zp) {
            const uint32_t b = p.zp[(long long)n * p.zrb + (g >> 1)];
            z = (g & 1) ? (int)(b >> 4) : (int)(b & 15u);
          }
          const long long si = (long long)n * p.G + g;
          const float s = p.scales_f16 ? __half2float(reinterpret_cast<const __half*>(p.scales)[si])
                                       : reinterpret_cast<const float*>(p.scales)[si];
          const uint32_t word = i < 8 ? wv.x : wv.y;
          v = __fmul_rn((float)((int)((word >> (4 * (i & 7))) & 15u) - z), s);
        } else {
          bad = true;
        }
        tile[16 * q + i][c] = v;
      }
      if (bad) report_status(p.status, kStatusBadIndex);
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
// Preparation.  One flat index space in three parts:
//   [0, N*K'/8)            one 32-bit word of 8 prepared codes (k' = 8w .. 8w+7 of row n);
//   next N*G'              one prepared scale, scales'[n, j] = scales[n, block_group[j]];
//   next N*ceil(G'/2)      one prepared zero-point byte (only when the weight has them).
// A padding slot (perm = -1) takes the block's zero point as its code, so its weight
// is exactly 0.  Indexes outside their range are not followed: they set
// kStatusBadIndex and write the zero-point code (or scale 0).
// ----------------------------------------------------------------------------------
struct PrepareArgs {
  const uint8_t* packed;
  const void* scales;
  const uint8_t* zp;
  int scales_f16;
  const int32_t* perm;
  const int32_t* bgroup;
  uint8_t* packed_out;
  void* scales_out;
  uint8_t* zp_out;
  int K, N, G, zrb, Kp, Gp, zrbp, bs;
  long long n_words, n_scales, n_total;
  uint32_t* status;
};

__device__ __forceinline__ uint32_t zp_of(const PrepareArgs& p, long long n, int g) {
  if (!p.zp) return 8u;
  const uint32_t b = p.zp[n * p.zrb + (g >> 1)];
  return (g & 1) ? (b >> 4) : (b & 15u);
}

__global__ void __launch_bounds__(256) act_order_prepare_kernel(const PrepareArgs p) {
  pdl_launch_dependents();
  pdl_wait();
  bool bad = false;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < p.n_total;
       idx += (long long)gridDim.x * blockDim.x) {
    if (idx < p.n_words) {
      const int wpr = p.Kp >> 3;
      const long long n = idx / wpr;
      const int k0 = (int)(idx - n * wpr) * 8;
      int g = p.bgroup[k0 / p.bs];
      if (g < 0 || g >= p.G) {
        bad = true;
        g = 0;
      }
      const uint32_t z = zp_of(p, n, g);
      const uint8_t* row = p.packed + n * (long long)(p.K >> 1);
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int src = p.perm[k0 + i];
        uint32_t c = z;
        if (src >= 0 && src < p.K) {
          c = nibble_at(row, src);
        } else if (src != -1) {
          bad = true;
        }
        word |= c << (4 * i);
      }
      *reinterpret_cast<uint32_t*>(p.packed_out + n * (long long)(p.Kp >> 1) + (k0 >> 1)) = word;
    } else if (idx < p.n_words + p.n_scales) {
      const long long e = idx - p.n_words;
      const long long n = e / p.Gp;
      const int j = (int)(e - n * p.Gp);
      const int g = p.bgroup[j];
      const bool ok = g >= 0 && g < p.G;
      bad |= !ok;
      if (p.scales_f16) {
        const uint16_t* s = reinterpret_cast<const uint16_t*>(p.scales);
        reinterpret_cast<uint16_t*>(p.scales_out)[e] = ok ? s[n * p.G + g] : (uint16_t)0;
      } else {
        const uint32_t* s = reinterpret_cast<const uint32_t*>(p.scales);
        reinterpret_cast<uint32_t*>(p.scales_out)[e] = ok ? s[n * p.G + g] : 0u;
      }
    } else {
      const long long e = idx - p.n_words - p.n_scales;
      const long long n = e / p.zrbp;
      const int b = (int)(e - n * p.zrbp);
      uint32_t v = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * b + h;
        if (j >= p.Gp) break;
        const int g = p.bgroup[j];
        const bool ok = g >= 0 && g < p.G;
        bad |= !ok;
        v |= (ok ? zp_of(p, n, g) : 0u) << (4 * h);
      }
      p.zp_out[e] = (uint8_t)v;
    }
  }
  if (bad) report_status(p.status, kStatusBadIndex);
}

// ----------------------------------------------------------------------------------
// Gather: out[m, k'] = A[m, perm[k']] (fp16 bits copied), +0 where perm[k'] = -1.  One
// thread writes 8 consecutive k' (16 bytes).  perm is constant for a weight, so it is
// read before the programmatic-launch wait; A only after it.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ void load_perm8(const int32_t* perm, int c, int (&src)[8]) {
  const int4 p0 = __ldg(reinterpret_cast<const int4*>(perm + 8 * c));
  const int4 p1 = __ldg(reinterpret_cast<const int4*>(perm + 8 * c + 4));
  src[0] = p0.x; src[1] = p0.y; src[2] = p0.z; src[3] = p0.w;
  src[4] = p1.x; src[5] = p1.y; src[6] = p1.z; src[7] = p1.w;
}

__global__ void __launch_bounds__(256) act_order_gather_kernel(const uint16_t* __restrict__ A,
                                                               const int32_t* __restrict__ perm,
                                                               uint16_t* __restrict__ out, int K, int Kp,
                                                               long long chunks, uint32_t* status) {
  pdl_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int cpr = Kp >> 3;
  int src[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
  if (idx < chunks) load_perm8(perm, (int)(idx % cpr), src);
  pdl_wait();
  bool bad = false;
  for (bool first = true; idx < chunks; idx += stride, first = false) {
    const long long m = idx / cpr;
    const int c = (int)(idx - m * cpr);
    if (!first) load_perm8(perm, c, src);
    const uint16_t* row = A + m * (long long)K;
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int s = src[i];
      h[i] = 0;
      if (s >= 0 && s < K) {
        h[i] = row[s];
      } else if (s != -1) {
        bad = true;
      }
    }
    *reinterpret_cast<uint4*>(out + m * (long long)Kp + 8 * c) =
        make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
  }
  if (bad) report_status(status, kStatusBadIndex);
}

}  // namespace

cudaError_t launch_dequant_gidx(LaunchCtx& ctx, const QWeight& w, const int32_t* gidx, int K, int N, int bs,
                                float* out) {
  DequantGidxArgs a = {};
  a.packed = w.packed;
  a.scales = w.scales;
  a.zp = w.zp;
  a.gidx = gidx;
  a.scales_f16 = w.scales_f16;
  a.out = out;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.status = ctx.status;
  const long long tiles = (long long)((N + 63) / 64) * ((K + 63) / 64);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ctx.variant = "dequant_gidx_f32_tile64";
  return launch_kernel(ctx, dequant_gidx_kernel, dim3((unsigned)tiles), dim3(256), 0, a);
}

cudaError_t launch_act_order_prepare(LaunchCtx& ctx, const QWeight& w, int K, int N, int bs, const int32_t* perm,
                                     const int32_t* bgroup, int Kp, uint8_t* packed_out, void* scales_out,
                                     uint8_t* zp_out) {
  PrepareArgs a = {};
  a.packed = w.packed;
  a.scales = w.scales;
  a.zp = w.zp;
  a.scales_f16 = w.scales_f16;
  a.perm = perm;
  a.bgroup = bgroup;
  a.packed_out = packed_out;
  a.scales_out = scales_out;
  a.zp_out = zp_out;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.Kp = Kp;
  a.Gp = Kp / bs;
  a.zrbp = (a.Gp + 1) / 2;
  a.bs = bs;
  a.n_words = (long long)N * (Kp / 8);
  a.n_scales = (long long)N * a.Gp;
  a.n_total = a.n_words + a.n_scales + (w.zp ? (long long)N * a.zrbp : 0);
  a.status = ctx.status;
  const long long blocks = (a.n_total + 255) / 256;
  const unsigned grid = (unsigned)(blocks < (long long)ctx.num_sms * 16 ? blocks : (long long)ctx.num_sms * 16);
  ctx.variant = "act_order_prepare";
  return launch_kernel(ctx, act_order_prepare_kernel, dim3(grid), dim3(256), 0, a);
}

cudaError_t launch_act_order_gather(LaunchCtx& ctx, const void* A, int M, int K, const int32_t* perm, int Kp,
                                    void* out) {
  const long long chunks = (long long)M * (Kp / 8);
  const long long blocks = (chunks + 255) / 256, cap = (long long)ctx.num_sms * 64;
  const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
  ctx.variant = "act_order_gather";
  return launch_kernel(ctx, act_order_gather_kernel, dim3(grid), dim3(256), 0,
                       static_cast<const uint16_t*>(A), perm, static_cast<uint16_t*>(out), K, Kp, chunks,
                       ctx.status);
}

}  // namespace mnb
