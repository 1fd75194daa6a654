// M = 1 decode GEMV over MatMulNBits int4 weights, the paired gate/up SwiGLU GEMV, and
// a generic CUDA-core kernel for shapes the fast kernels do not take.
//
// Fast GEMV design (one GB300: 152 SMs, HBM-bound):
//   * A CTA owns a contiguous range of output columns (a static grid of 1-2 CTAs per SM,
//     columns split evenly), so every weight row it reads is one contiguous byte range.
//   * K is cut into 32-element chunks (16 bytes of nibbles).  Thread s of the CTA owns
//     chunks s, s + S, s + 2S, ... (S = threads per CTA) of every column, so each warp
//     load instruction reads 512 contiguous bytes of one row with 128-bit loads.
//   * The thread keeps the activations of its chunks in registers for the whole kernel
//     (A is read once per CTA), pre-paired to match the nibble conversion below.
//   * Weights stream through a two-deep register pipeline of column batches.  The first
//     batch is requested before the programmatic-launch wait, so a kernel launched behind
//     another one streams its weights while the previous kernel finishes.
//   * Each chunk's nibbles become exact fp16 (code - zp) (magic-number conversion), the
//     32-term partial dot with the activations is formed with exact fp16 x fp16 products
//     summed in fp32, and then multiplied by the chunk's group scale (the scale is
//     applied after the partial dot, as in matmul_nbits_gemv_f16 of matmul_nbits.rs; a
//     group of 64 or 128 is the sum of its 32-element partials, each scaled by the same
//     group scale).
//   * Per-column partials are reduced across the warp with a transposed butterfly and
//     across warps in shared memory, in a fixed order (deterministic), then rounded once
//     to fp16.
#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int kMaxColsPerCta = 64;

struct GemvArgs {
  const __half* A;
  const uint8_t* packed[2];
  const void* scales[2];
  const uint8_t* zp[2];
  int scales_f16[2];
  void* Y;
  int K, N, G, zrb;
  int group_shift;  // log2(bs / 32) when bs >= 32
  const __half* bias;
  int bias_mode;
};

__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

// Partial dot of one 32-bit word of eight nibbles (natural order) with four pre-paired
// activation half2 registers: exact products, fp32 sums.
__device__ __forceinline__ float dot_word(uint32_t w, uint32_t zlo, uint32_t zhi,
                                          const uint32_t* a, float acc) {
  uint32_t d[4];
  nibbles_to_centered_half2(w, zlo, zhi, d);
  acc = fma2_f16_f32(d[0], a[0], acc);
  acc = fma2_f16_f32(d[1], a[1], acc);
  acc = fma2_f16_f32(d[2], a[2], acc);
  acc = fma2_f16_f32(d[3], a[3], acc);
  return acc;
}

template <int NW, int CPS, int CB, bool BS16, bool PAIR>
__global__ void __launch_bounds__(NW * 32, (NW == 1 ? 16 : (NW == 4 ? 4 : (NW == 8 ? 2 : 1))))
    gemv_kernel(const GemvArgs p) {
  constexpr int S = NW * 32;
  constexpr int NWT = PAIR ? 2 : 1;
  constexpr int V = CB * NWT;  // values reduced per batch
  constexpr int kLog2V = (V == 1) ? 0 : (V == 2) ? 1 : (V == 4) ? 2 : (V == 8) ? 3 : (V == 16) ? 4 : 5;
  constexpr int kNS = BS16 ? 2 : 1;  // scales per chunk
  __shared__ float red[NW][NWT][kMaxColsPerCta];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = p.K >> 5;
  const int n0 = (int)(((long long)blockIdx.x * p.N) / gridDim.x);
  const int n1 = (int)(((long long)(blockIdx.x + 1) * p.N) / gridDim.x);
  const long long row_bytes = p.K >> 1;

  uint4 wv[2][CB][NWT][CPS];
  uint32_t sraw[2][CB][NWT][CPS][kNS];
  uint32_t zraw[2][CB][NWT][CPS];

  auto load_batch = [&](const int buf, const int nb) {
#pragma unroll
    for (int i = 0; i < CB; ++i) {
      const int n = nb + i;
      const bool colok = n < n1;
#pragma unroll
      for (int t = 0; t < NWT; ++t) {
        const uint8_t* prow = p.packed[t] + (long long)n * row_bytes;
#pragma unroll
        for (int j = 0; j < CPS; ++j) {
          const int c = tid + j * S;
          const bool ok = colok && c < C;
          wv[buf][i][t][j] = ok ? ld_stream_v4(prow + (long long)c * 16) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int e = 0; e < kNS; ++e) {
            const int g = BS16 ? (2 * c + e) : (c >> p.group_shift);
            const long long si = (long long)n * p.G + g;
            uint32_t s = 0;
            if (ok) s = p.scales_f16[t] ? ld_nc_u16((const uint16_t*)p.scales[t] + si)
                                        : ld_nc_u32((const uint32_t*)p.scales[t] + si);
            sraw[buf][i][t][j][e] = s;
          }
          const int zb = BS16 ? c : ((c >> p.group_shift) >> 1);
          zraw[buf][i][t][j] =
              (ok && p.zp[t]) ? ld_nc_u8(p.zp[t] + (long long)n * p.zrb + zb) : 0x88u;
        }
      }
    }
  };

  // Activations of this thread's chunks, paired for the conversion order.
  uint32_t a[CPS][16];

  auto compute_batch = [&](const int buf, const int nb) {
    float part[V];
#pragma unroll
    for (int i = 0; i < CB; ++i) {
#pragma unroll
      for (int t = 0; t < NWT; ++t) {
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < CPS; ++j) {
          const int c = tid + j * S;
          if (c < C) {
            const uint4 w4 = wv[buf][i][t][j];
            const uint32_t z = zraw[buf][i][t][j];
            if (BS16) {
              const uint32_t z0 = z & 15u, z1 = (z >> 4) & 15u;
              float p0 = dot_word(w4.x, zp_lo_const(z0), zp_hi_const(z0), &a[j][0], 0.0f);
              p0 = dot_word(w4.y, zp_lo_const(z0), zp_hi_const(z0), &a[j][4], p0);
              float p1 = dot_word(w4.z, zp_lo_const(z1), zp_hi_const(z1), &a[j][8], 0.0f);
              p1 = dot_word(w4.w, zp_lo_const(z1), zp_hi_const(z1), &a[j][12], p1);
              const float s0 = p.scales_f16[t] ? half_bits_to_float(sraw[buf][i][t][j][0])
                                               : __uint_as_float(sraw[buf][i][t][j][0]);
              const float s1 = p.scales_f16[t] ? half_bits_to_float(sraw[buf][i][t][j][kNS - 1])
                                               : __uint_as_float(sraw[buf][i][t][j][kNS - 1]);
              acc = fmaf(p0, s0, acc);
              acc = fmaf(p1, s1, acc);
            } else {
              const int g = c >> p.group_shift;
              const uint32_t zz = (g & 1) ? ((z >> 4) & 15u) : (z & 15u);
              const uint32_t zlo = zp_lo_const(zz), zhi = zp_hi_const(zz);
              float q0 = dot_word(w4.x, zlo, zhi, &a[j][0], 0.0f);
              float q1 = dot_word(w4.y, zlo, zhi, &a[j][4], 0.0f);
              q0 = dot_word(w4.z, zlo, zhi, &a[j][8], q0);
              q1 = dot_word(w4.w, zlo, zhi, &a[j][12], q1);
              const float s = p.scales_f16[t] ? half_bits_to_float(sraw[buf][i][t][j][0])
                                              : __uint_as_float(sraw[buf][i][t][j][0]);
              acc = fmaf(q0 + q1, s, acc);
            }
          }
        }
        part[i * NWT + t] = acc;
      }
    }
    const float r = warp_transpose_reduce<V>(part, lane);
    if ((lane & ((32 >> kLog2V) - 1)) == 0) {
      const int v = lane >> (5 - kLog2V);
      const int i = v / NWT, t = v % NWT;
      const int col = nb + i;
      if (col < n1) red[warp][t][col - n0] = r;
    }
  };

  // Weights first (no earlier kernel writes them), then wait for A's producer.
  if (n0 < n1) load_batch(0, n0);
  pdl_launch_dependents();
  pdl_wait();

#pragma unroll
  for (int j = 0; j < CPS; ++j) {
    const int c = tid + j * S;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 x = make_uint4(0, 0, 0, 0);
      if (c < C) x = *reinterpret_cast<const uint4*>(p.A + (long long)c * 32 + q * 8);
      pair_halves_stride4(x, &a[j][q * 4]);
    }
  }

  for (int nb = n0; nb < n1; nb += 2 * CB) {
    if (nb + CB < n1) load_batch(1, nb + CB);
    compute_batch(0, nb);
    if (nb + CB < n1) {
      if (nb + 2 * CB < n1) load_batch(0, nb + 2 * CB);
      compute_batch(1, nb + CB);
    }
  }
  __syncthreads();

  for (int c = tid; c < n1 - n0; c += S) {
    float v[NWT];
#pragma unroll
    for (int t = 0; t < NWT; ++t) {
      float s = 0.0f;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += red[w][t][c];
      v[t] = s;
    }
    __half out;
    if (PAIR) out = __float2half_rn(silu_f32(v[0]) * v[NWT - 1]);
    else out = round_out(v[0], p.bias, n0 + c, p.bias_mode);
    reinterpret_cast<__half*>(p.Y)[n0 + c] = out;
  }
}

// ----------------------------------------------------------------------------------
// Generic kernel: any M (8-row tiles on grid.y), any K % 16 == 0, any block size.
// One warp per output column; lanes stride over 16-element pieces of K; fp32 math.
// ----------------------------------------------------------------------------------
struct GenericArgs {
  const __half* A;
  const uint8_t* packed[2];
  const void* scales[2];
  const uint8_t* zp[2];
  int scales_f16[2];
  void* Y;
  int M, K, N, G, zrb, bs;
  const __half* bias;
  int bias_mode;
};

template <bool PAIR>
__global__ void __launch_bounds__(256) generic_kernel(const GenericArgs p) {
  constexpr int NWT = PAIR ? 2 : 1;
  constexpr int R = 8;  // rows per tile
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = blockIdx.x * 8 + warp;
  const int m0 = blockIdx.y * R;
  pdl_launch_dependents();
  pdl_wait();
  if (n >= p.N) return;
  const long long row_bytes = p.K >> 1;
  const int pieces = p.K >> 4;
  float acc[NWT][R];
#pragma unroll
  for (int t = 0; t < NWT; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[t][r] = 0.0f;

  for (int pc = lane; pc < pieces; pc += 32) {
    const int k0 = pc * 16;
    const int g = k0 / p.bs;
    float w[NWT][16];
    float sc[NWT];
#pragma unroll
    for (int t = 0; t < NWT; ++t) {
      const uint2 wv = *reinterpret_cast<const uint2*>(p.packed[t] + (long long)n * row_bytes + pc * 8);
      int z = 8;
      if (p.zp[t]) {
        const uint32_t b = p.zp[t][(long long)n * p.zrb + (g >> 1)];
        z = (g & 1) ? (int)(b >> 4) : (int)(b & 15u);
      }
      const long long si = (long long)n * p.G + g;
      sc[t] = p.scales_f16[t] ? __half2float(reinterpret_cast<const __half*>(p.scales[t])[si])
                              : reinterpret_cast<const float*>(p.scales[t])[si];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        w[t][i] = (float)((int)((wv.x >> (4 * i)) & 15u) - z);
        w[t][8 + i] = (float)((int)((wv.y >> (4 * i)) & 15u) - z);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int m = m0 + r;
      if (m < p.M) {
        const __half* arow = p.A + (long long)m * p.K + k0;
        const uint4 x0 = *reinterpret_cast<const uint4*>(arow);
        const uint4 x1 = *reinterpret_cast<const uint4*>(arow + 8);
        const __half* h0 = reinterpret_cast<const __half*>(&x0);
        const __half* h1 = reinterpret_cast<const __half*>(&x1);
#pragma unroll
        for (int t = 0; t < NWT; ++t) {
          float d = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) d = fmaf(w[t][i], __half2float(h0[i]), d);
#pragma unroll
          for (int i = 0; i < 8; ++i) d = fmaf(w[t][8 + i], __half2float(h1[i]), d);
          acc[t][r] = fmaf(d, sc[t], acc[t][r]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NWT; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) acc[t][r] += __shfl_xor_sync(kFull, acc[t][r], o);
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int m = m0 + r;
      if (m < p.M) {
        __half out;
        if (PAIR) out = __float2half_rn(silu_f32(acc[0][r]) * acc[NWT - 1][r]);
        else out = round_out(acc[0][r], p.bias, n, p.bias_mode);
        reinterpret_cast<__half*>(p.Y)[(long long)m * p.N + n] = out;
      }
    }
  }
}

// ----------------------------------------------------------------------------------
// Host planning
// ----------------------------------------------------------------------------------
struct GemvPlan {
  int nw, cps, ctas_per_sm;
  bool ok;
};

GemvPlan plan_gemv(int K) {
  if (K % 32 != 0) return {0, 0, 0, false};
  const int C = K / 32;
  if (C <= 32) return {1, 1, 8, true};
  if (C <= 128) return {4, 1, 2, true};
  if (C <= 256) return {8, 1, 1, true};
  if (C <= 512) return {8, 2, 1, true};
  if (C <= 1024) return {16, 2, 1, true};
  return {0, 0, 0, false};
}

template <bool PAIR>
using GemvKernelPtr = void (*)(const GemvArgs);

template <int NW, int CPS, bool PAIR>
GemvKernelPtr<PAIR> pick_cb(bool bs16) {
  // Four 16-byte weight loads per thread per batch, two batches in flight.
  constexpr int NWT = PAIR ? 2 : 1;
  constexpr int L = 4;
  constexpr int CB0 = L / (NWT * CPS);
  constexpr int CB = CB0 < 1 ? 1 : CB0;
  return bs16 ? gemv_kernel<NW, CPS, CB, true, PAIR> : gemv_kernel<NW, CPS, CB, false, PAIR>;
}

template <bool PAIR>
GemvKernelPtr<PAIR> select_gemv(const GemvPlan& pl, bool bs16) {
  if (pl.nw == 1) return pick_cb<1, 1, PAIR>(bs16);
  if (pl.nw == 4) return pick_cb<4, 1, PAIR>(bs16);
  if (pl.nw == 8 && pl.cps == 1) return pick_cb<8, 1, PAIR>(bs16);
  if (pl.nw == 8) return pick_cb<8, 2, PAIR>(bs16);
  return pick_cb<16, 2, PAIR>(bs16);
}

int log2_int(int v) {
  int r = 0;
  while ((1 << r) < v) ++r;
  return r;
}

template <bool PAIR>
cudaError_t launch_gemv_impl(LaunchCtx& ctx, const void* A, const QWeight* w, int K, int N,
                             int bs, void* Y) {
  const GemvPlan pl = plan_gemv(K);
  if (!pl.ok) return cudaErrorNotSupported;
  GemvArgs a = {};
  a.A = static_cast<const __half*>(A);
  const int nwt = PAIR ? 2 : 1;
  for (int t = 0; t < 2; ++t) {
    const QWeight& q = w[t < nwt ? t : 0];
    a.packed[t] = q.packed;
    a.scales[t] = q.scales;
    a.zp[t] = q.zp;
    a.scales_f16[t] = q.scales_f16;
  }
  a.Y = Y;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.group_shift = bs >= 32 ? log2_int(bs / 32) : 0;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = PAIR ? 0 : ctx.bias_mode;
  long long grid = (long long)ctx.num_sms * pl.ctas_per_sm;
  if (grid > N) grid = N;
  const long long min_grid = (N + kMaxColsPerCta - 1) / kMaxColsPerCta;
  if (grid < min_grid) grid = min_grid;
  auto kern = select_gemv<PAIR>(pl, bs == 16);
  ctx.variant = PAIR ? "gemv_pair_swiglu_f16acc32" : "gemv_f16acc32";
  return launch_kernel(ctx, kern, dim3((unsigned)grid), dim3(pl.nw * 32), 0, a);
}

template <bool PAIR>
cudaError_t launch_generic_impl(LaunchCtx& ctx, const void* A, int M, const QWeight* w, int K,
                                int N, int bs, void* Y) {
  GenericArgs a = {};
  a.A = static_cast<const __half*>(A);
  const int nwt = PAIR ? 2 : 1;
  for (int t = 0; t < 2; ++t) {
    const QWeight& q = w[t < nwt ? t : 0];
    a.packed[t] = q.packed;
    a.scales[t] = q.scales;
    a.zp[t] = q.zp;
    a.scales_f16[t] = q.scales_f16;
  }
  a.Y = Y;
  a.M = M;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.bs = bs;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = PAIR ? 0 : ctx.bias_mode;
  dim3 grid((N + 7) / 8, (M + 7) / 8);
  ctx.variant = PAIR ? "generic_pair_swiglu" : "generic";
  return launch_kernel(ctx, generic_kernel<PAIR>, grid, dim3(256), 0, a);
}

}  // namespace

cudaError_t launch_gemv(LaunchCtx& ctx, const void* A, const QWeight& w, int K, int N, int bs,
                        void* Y) {
  return launch_gemv_impl<false>(ctx, A, &w, K, N, bs, Y);
}

cudaError_t launch_gemv_pair_swiglu(LaunchCtx& ctx, const void* A, const QWeight& gate,
                                    const QWeight& up, int K, int N, int bs, void* out) {
  const QWeight w[2] = {gate, up};
  return launch_gemv_impl<true>(ctx, A, w, K, N, bs, out);
}

cudaError_t launch_generic(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N,
                           int bs, void* Y) {
  return launch_generic_impl<false>(ctx, A, M, &w, K, N, bs, Y);
}

cudaError_t launch_generic_pair_swiglu(LaunchCtx& ctx, const void* A, const QWeight& gate,
                                       const QWeight& up, int K, int N, int bs, void* out) {
  const QWeight w[2] = {gate, up};
  return launch_generic_impl<true>(ctx, A, 1, w, K, N, bs, out);
}

}  // namespace mnb
