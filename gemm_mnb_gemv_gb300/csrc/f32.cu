// fp32 activations: Y[M,N] = A[M,K] . dequant(B)^T with fp32 A, Y and bias, the
// operator's fp32 path (matmul_nbits.rs: MatMulNBitsKernel::run with a Float32 A, the
// matmul_nbits_gemv_f32 kernel for M = 1 and dequantise-then-GEMM otherwise).
//
// M = 1 runs the bulk-copy GEMV with fp32 activations in registers (gemv_tma.cu).  For
// M >= 2 the tensor cores take fp16 operands, so each fp32 row is split exactly enough:
// with e = the row's binary exponent (max |a| < 2^(e + 15)), x = a * 2^-e,
//   hi = fp16(x), lo = fp16(x - hi),   |x - (hi + lo)| <= 2^-22 |x|,
// and the two become rows 2m and 2m + 1 of an fp16 activation matrix.  The GEMM kernels
// (gemm_smallm.cu, gemm_tc.cu) then add the two accumulator rows of each pair and scale
// by 2^e in fp32.  The weights are exact in fp16 ((code - zp), scale applied to the fp32
// accumulator), so the only extra error is the 2^-22 split, far below fp16 rounding.
#include <cfloat>

#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

// One CTA per row: the row maximum, its exponent, then the hi/lo rows.
__global__ void __launch_bounds__(256) split_rows_kernel(const float* __restrict__ A, __half* __restrict__ A2,
                                                         int* __restrict__ rexp, int K) {
  __shared__ float wmax[8];
  __shared__ int e_sh;
  pdl_launch_dependents();
  pdl_wait();
  const long long m = blockIdx.x;
  const float* row = A + m * K;
  float mx = 0.0f;
  for (int k = threadIdx.x * 4; k < K; k += 256 * 4) {  // K % 16 == 0
    const float4 v = *reinterpret_cast<const float4*>(row + k);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = wmax[0];
    for (int i = 1; i < 8; ++i) r = fmaxf(r, wmax[i]);
    int e = 0;
    if (r > 0.0f && r <= FLT_MAX) {
      int E;
      (void)frexpf(r, &E);  // r < 2^E
      e = E - 15;           // so max |x| < 2^15
    }
    e_sh = e;
    rexp[m] = e;
  }
  __syncthreads();
  const int e = e_sh;
  __half* hi = A2 + (2 * m) * (long long)K;
  __half* lo = hi + K;
  for (int k = threadIdx.x * 8; k < K; k += 256 * 8) {
    const float4 v0 = *reinterpret_cast<const float4*>(row + k);
    const float4 v1 = *reinterpret_cast<const float4*>(row + k + 4);
    const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float x0 = ldexpf(x[2 * i], -e), x1 = ldexpf(x[2 * i + 1], -e);
      const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
      const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
      h[i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      l[i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
    }
    *reinterpret_cast<uint4*>(hi + k) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + k) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// Generic fp32 kernel: any M (8-row tiles on grid.y), any K % 16 == 0, any block size.
// One warp per output column; lanes stride over 16-element pieces of K.
struct GenericF32Args {
  const float* A;
  const uint8_t* packed;
  const void* scales;
  const uint8_t* zp;
  int scales_f16;
  float* Y;
  const float* bias;
  int M, K, N, G, zrb, bs;
};

__global__ void __launch_bounds__(256) generic_f32_kernel(const GenericF32Args p) {
  constexpr int R = 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = blockIdx.x * 8 + warp;
  const int m0 = blockIdx.y * R;
  pdl_launch_dependents();
  pdl_wait();
  if (n >= p.N) return;
  const long long row_bytes = p.K >> 1;
  float acc[R];
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.0f;
  for (int pc = lane; pc < (p.K >> 4); pc += 32) {
    const int k0 = pc * 16;
    const int g = k0 / p.bs;
    const uint2 wv = *reinterpret_cast<const uint2*>(p.packed + (long long)n * row_bytes + pc * 8);
    int z = 8;
    if (p.zp) {
      const uint32_t b = p.zp[(long long)n * p.zrb + (g >> 1)];
      z = (g & 1) ? (int)(b >> 4) : (int)(b & 15u);
    }
    const long long si = (long long)n * p.G + g;
    const float sc = p.scales_f16 ? __half2float(reinterpret_cast<const __half*>(p.scales)[si])
                                  : reinterpret_cast<const float*>(p.scales)[si];
    float w[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      w[i] = (float)((int)((wv.x >> (4 * i)) & 15u) - z);
      w[8 + i] = (float)((int)((wv.y >> (4 * i)) & 15u) - z);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int m = m0 + r;
      if (m < p.M) {
        const float* arow = p.A + (long long)m * p.K + k0;
        float d = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 x = *reinterpret_cast<const float4*>(arow + 4 * q);
          d = fmaf(w[4 * q], x.x, d);
          d = fmaf(w[4 * q + 1], x.y, d);
          d = fmaf(w[4 * q + 2], x.z, d);
          d = fmaf(w[4 * q + 3], x.w, d);
        }
        acc[r] = fmaf(d, sc, acc[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc[r] += __shfl_xor_sync(kFull, acc[r], o);
  if (lane == 0) {
    const float b = p.bias ? p.bias[n] : 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int m = m0 + r;
      if (m < p.M) p.Y[(long long)m * p.N + n] = acc[r] + b;
    }
  }
}

}  // namespace

cudaError_t launch_split_f32(LaunchCtx& ctx, const float* A, int M, int K, void* A2, int* rexp) {
  ctx.variant = "split_f32_rows";
  return launch_kernel(ctx, split_rows_kernel, dim3((unsigned)M), dim3(256), 0, A, static_cast<__half*>(A2), rexp,
                       K);
}

cudaError_t launch_generic_f32(LaunchCtx& ctx, const float* A, int M, const QWeight& w, int K, int N, int bs,
                               float* Y, const float* bias) {
  GenericF32Args a = {};
  a.A = A;
  a.packed = w.packed;
  a.scales = w.scales;
  a.zp = w.zp;
  a.scales_f16 = w.scales_f16;
  a.Y = Y;
  a.bias = bias;
  a.M = M;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.bs = bs;
  const long long gy = (M + 7) / 8;
  if (gy > 65535) return cudaErrorNotSupported;
  ctx.variant = "generic_f32";
  return launch_kernel(ctx, generic_f32_kernel, dim3((N + 7) / 8, (unsigned)gy), dim3(256), 0, a);
}

}  // namespace mnb
