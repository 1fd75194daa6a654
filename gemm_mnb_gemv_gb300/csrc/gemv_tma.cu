// M = 1 GEMV (and the paired gate/up SwiGLU GEMV) with a bulk-copy (TMA) ring.
//
// A CTA owns a contiguous range of output columns, so its packed weights, scales and
// zero points are three contiguous byte ranges of the MatMulNBits storage.  One producer
// lane streams them, a stage of CB columns at a time, with 1-D `cp.async.bulk` copies
// into a ring of shared-memory slots (64-100 KB in flight per SM, independent of the
// register budget).  Eight consumer warps keep their activations in registers, read each
// stage's 16-byte weight chunks from shared memory, form exact fp16 (code - zp) with the
// magic-number conversion, accumulate exact fp16 x fp16 products in fp32, apply the group
// scale to each 32-element partial dot, and reduce per column in a fixed order.
//
// Warps are grouped: WG consumer warps cover one column's K range (lane slot s owns the
// 32-element chunks s, s + 32 WG, ...), and 8 / WG groups work on different columns of a
// stage.  Every wait on an mbarrier is bounded; a wait that gives up records its cause in
// the device status word and the kernel finishes without further shared-memory traffic
// (its outputs are then NaN).
//
// The producer issues its copies before the programmatic-launch wait (the weights are
// never written by the preceding kernel); consumers wait before reading A.
#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxColsPerCta = 128;
constexpr int kMaxStages = 8;
constexpr int kRingBudget = 100 * 1024;

struct TmaGemvArgs {
  const __half* A;
  const uint8_t* packed[2];
  const uint8_t* scales[2];
  const uint8_t* zp[2];
  int scales_f16[2];
  void* Y;
  int K, N, G;
  int group_shift;
  int row_bytes;   // K / 2
  int sbytes[2];   // scale bytes per row
  int zbytes[2];   // zero-point bytes per row (0 when absent)
  int stage_bytes;
  int stages;
  uint32_t* status;
};

__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float dot_word_tma(uint32_t w, uint32_t zlo, uint32_t zhi,
                                              const uint32_t* a, float acc) {
  uint32_t d[4];
  nibbles_to_centered_half2(w, zlo, zhi, d);
  acc = fma2_f16_f32(d[0], a[0], acc);
  acc = fma2_f16_f32(d[1], a[1], acc);
  acc = fma2_f16_f32(d[2], a[2], acc);
  acc = fma2_f16_f32(d[3], a[3], acc);
  return acc;
}

template <int WG, int CPS, int VPG, bool BS16, bool PAIR>
__global__ void __launch_bounds__(kThreads, 2) gemv_tma_kernel(const TmaGemvArgs p) {
  constexpr int NG = kConsumerWarps / WG;
  constexpr int CB = NG * VPG;
  constexpr int NWT = PAIR ? 2 : 1;
  constexpr int V = VPG * NWT;
  constexpr int kLog2V = (V == 1) ? 0 : (V == 2) ? 1 : (V == 4) ? 2 : (V == 8) ? 3 : 4;
  static_assert(V <= 16, "too many values per lane");

  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full_bar[kMaxStages];
  __shared__ uint64_t empty_bar[kMaxStages];
  __shared__ float red[WG][NWT][kMaxColsPerCta];
  __shared__ int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = (int)(((long long)blockIdx.x * p.N) / gridDim.x);
  const int n1 = (int)(((long long)(blockIdx.x + 1) * p.N) / gridDim.x);
  const int nstages_total = (n1 - n0 + CB - 1) / CB;
  const int S = p.stages;
  const int C = p.K >> 5;

  // Region offsets inside a stage: for each weight, packed | scales | zero points.
  int off_p[NWT], off_s[NWT], off_z[NWT];
  {
    int off = 0;
#pragma unroll
    for (int t = 0; t < NWT; ++t) {
      off_p[t] = off;
      off += CB * p.row_bytes;
      off_s[t] = off;
      off += CB * p.sbytes[t];
      off_z[t] = off;
      off += CB * p.zbytes[t];
    }
  }

  if (tid == 0) {
    failed = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------- producer -------------------------------------
    int issued = 0;
    if (lane == 0) {
      for (int st = 0; st < nstages_total; ++st) {
        const int slot = st % S;
        const uint32_t round = (uint32_t)(st / S);
        if (st >= S && !mbar_wait_bounded(&empty_bar[slot], (round - 1) & 1u)) {
          report_status(p.status, kStatusEmptyWait);
          atomicExch(&failed, 1);
          break;
        }
        const int col = n0 + st * CB;
        const int nc = min(CB, n1 - col);
        uint32_t bytes = 0;
#pragma unroll
        for (int t = 0; t < NWT; ++t) bytes += (uint32_t)nc * (p.row_bytes + p.sbytes[t] + p.zbytes[t]);
        uint8_t* base = ring + (size_t)slot * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], bytes);
#pragma unroll
        for (int t = 0; t < NWT; ++t) {
          bulk_g2s(base + off_p[t], p.packed[t] + (long long)col * p.row_bytes, nc * p.row_bytes,
                   &full_bar[slot]);
          bulk_g2s(base + off_s[t], p.scales[t] + (long long)col * p.sbytes[t], nc * p.sbytes[t],
                   &full_bar[slot]);
          if (p.zbytes[t])
            bulk_g2s(base + off_z[t], p.zp[t] + (long long)col * p.zbytes[t], nc * p.zbytes[t],
                     &full_bar[slot]);
        }
        issued = st + 1;
      }
    }
    // Every copy this lane issued must land before the CTA can exit.  Consumers have
    // normally waited for all of them already; after a failed wait this bounds the drain.
    if (lane == 0) {
      for (int st = issued > S ? issued - S : 0; st < issued; ++st)
        (void)mbar_wait_bounded(&full_bar[st % S], (uint32_t)(st / S) & 1u);
    }
    pdl_launch_dependents();
  } else {
    // ------------------------------- consumers ------------------------------------
    pdl_launch_dependents();
    pdl_wait();
    const int g = warp / WG, wig = warp % WG;
    const int ls = wig * 32 + lane;

    uint32_t a[CPS][16];
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      const int c = ls + j * WG * 32;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 x = make_uint4(0, 0, 0, 0);
        if (c < C) x = *reinterpret_cast<const uint4*>(p.A + (long long)c * 32 + q * 8);
        pair_halves_stride4(x, &a[j][q * 4]);
      }
    }

    bool ok = true;
    for (int st = 0; st < nstages_total; ++st) {
      const int slot = st % S;
      const uint32_t round = (uint32_t)(st / S);
      if (ok && !mbar_wait_bounded(&full_bar[slot], round & 1u)) {
        report_status(p.status, kStatusFullWait);
        atomicExch(&failed, 1);
        ok = false;
      }
      const int col0 = n0 + st * CB;
      const int nc = min(CB, n1 - col0);
      const uint8_t* base = ring + (size_t)slot * p.stage_bytes;
      float part[V];
#pragma unroll
      for (int vi = 0; vi < VPG; ++vi) {
        const int ci = g + vi * NG;
#pragma unroll
        for (int t = 0; t < NWT; ++t) {
          float acc = 0.0f;
          if (ok && ci < nc) {
            const uint8_t* pp = base + off_p[t] + ci * p.row_bytes;
            const uint8_t* ps = base + off_s[t] + ci * p.sbytes[t];
            const uint8_t* pz = base + off_z[t] + ci * p.zbytes[t];
#pragma unroll
            for (int j = 0; j < CPS; ++j) {
              const int c = ls + j * WG * 32;
              if (c < C) {
                const uint4 w4 = lds128(pp + c * 16);
                if (BS16) {
                  const uint32_t zb = p.zbytes[t] ? (uint32_t)pz[c] : 0x88u;
                  const uint32_t z0 = zb & 15u, z1 = zb >> 4;
                  const uint32_t zl0 = zp_lo_const(z0), zh0 = zp_hi_const(z0);
                  const uint32_t zl1 = zp_lo_const(z1), zh1 = zp_hi_const(z1);
                  float p0 = dot_word_tma(w4.x, zl0, zh0, &a[j][0], 0.0f);
                  p0 = dot_word_tma(w4.y, zl0, zh0, &a[j][4], p0);
                  float p1 = dot_word_tma(w4.z, zl1, zh1, &a[j][8], 0.0f);
                  p1 = dot_word_tma(w4.w, zl1, zh1, &a[j][12], p1);
                  float s0, s1;
                  if (p.scales_f16[t]) {
                    const __half* sh = reinterpret_cast<const __half*>(ps);
                    s0 = __half2float(sh[2 * c]);
                    s1 = __half2float(sh[2 * c + 1]);
                  } else {
                    const float* sf = reinterpret_cast<const float*>(ps);
                    s0 = sf[2 * c];
                    s1 = sf[2 * c + 1];
                  }
                  acc = fmaf(p0, s0, acc);
                  acc = fmaf(p1, s1, acc);
                } else {
                  const int gi = c >> p.group_shift;
                  uint32_t zz = 8u;
                  if (p.zbytes[t]) {
                    const uint32_t zb = pz[gi >> 1];
                    zz = (gi & 1) ? (zb >> 4) : (zb & 15u);
                  }
                  const uint32_t zlo = zp_lo_const(zz), zhi = zp_hi_const(zz);
                  float q0 = dot_word_tma(w4.x, zlo, zhi, &a[j][0], 0.0f);
                  float q1 = dot_word_tma(w4.y, zlo, zhi, &a[j][4], 0.0f);
                  q0 = dot_word_tma(w4.z, zlo, zhi, &a[j][8], q0);
                  q1 = dot_word_tma(w4.w, zlo, zhi, &a[j][12], q1);
                  const float s = p.scales_f16[t]
                                      ? __half2float(reinterpret_cast<const __half*>(ps)[gi])
                                      : reinterpret_cast<const float*>(ps)[gi];
                  acc = fmaf(q0 + q1, s, acc);
                }
              }
            }
          }
          part[vi * NWT + t] = acc;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp no longer reads the slot
      const float r = warp_transpose_reduce<V>(part, lane);
      if ((lane & ((32 >> kLog2V) - 1)) == 0) {
        const int v = lane >> (5 - kLog2V);
        const int vi = v / NWT, t = v % NWT;
        const int ci = g + vi * NG;
        if (ci < nc) red[wig][t][st * CB + ci] = r;
      }
    }
  }
  __syncthreads();

  const bool bad = failed != 0;
  for (int c = tid; c < n1 - n0; c += kThreads) {
    float v[NWT];
#pragma unroll
    for (int t = 0; t < NWT; ++t) {
      float s = 0.0f;
#pragma unroll
      for (int w = 0; w < WG; ++w) s += red[w][t][c];
      v[t] = s;
    }
    float o = PAIR ? silu_f32(v[0]) * v[NWT - 1] : v[0];
    if (bad) o = __int_as_float(0x7fc00000);
    reinterpret_cast<__half*>(p.Y)[n0 + c] = __float2half_rn(o);
  }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
template <bool PAIR>
using TmaKernel = void (*)(const TmaGemvArgs);

template <int WG, int CPS, bool PAIR>
TmaKernel<PAIR> pick(bool bs16) {
  constexpr int VPG = PAIR ? 2 : 4;
  return bs16 ? gemv_tma_kernel<WG, CPS, VPG, true, PAIR> : gemv_tma_kernel<WG, CPS, VPG, false, PAIR>;
}

template <bool PAIR>
TmaKernel<PAIR> select_kernel(int wg, int cps, bool bs16) {
  if (wg == 1) return pick<1, 1, PAIR>(bs16);
  if (wg == 2) return pick<2, 1, PAIR>(bs16);
  if (wg == 4) return pick<4, 1, PAIR>(bs16);
  if (cps == 1) return pick<8, 1, PAIR>(bs16);
  if (cps == 2) return pick<8, 2, PAIR>(bs16);
  return pick<8, 4, PAIR>(bs16);
}

template <bool PAIR>
cudaError_t launch_tma_impl(LaunchCtx& ctx, const void* A, const QWeight* w, int K, int N, int bs,
                            void* Y) {
  constexpr int NWT = PAIR ? 2 : 1;
  if (K % 32 != 0) return cudaErrorNotSupported;
  const int C = K / 32;
  int wg = 1;
  while (wg < 8 && wg * 32 < C) wg *= 2;
  int cps = (C + wg * 32 - 1) / (wg * 32);
  if (cps == 3) cps = 4;
  if (cps > 4) return cudaErrorNotSupported;
  const int ng = kConsumerWarps / wg;
  const int cb = ng * (PAIR ? 2 : 4);
  const int G = K / bs;
  TmaGemvArgs a = {};
  a.A = static_cast<const __half*>(A);
  a.Y = Y;
  a.K = K;
  a.N = N;
  a.G = G;
  a.row_bytes = K / 2;
  a.group_shift = 0;
  while (bs >= 32 && (32 << a.group_shift) < bs) ++a.group_shift;
  int col_bytes = 0;
  for (int t = 0; t < 2; ++t) {
    const QWeight& q = w[t < NWT ? t : 0];
    a.packed[t] = q.packed;
    a.scales[t] = static_cast<const uint8_t*>(q.scales);
    a.zp[t] = q.zp;
    a.scales_f16[t] = q.scales_f16;
    a.sbytes[t] = G * (q.scales_f16 ? 2 : 4);
    a.zbytes[t] = q.zp ? (G + 1) / 2 : 0;
    if (t < NWT) {
      if (a.sbytes[t] % 16 != 0 || a.zbytes[t] % 16 != 0) return cudaErrorNotSupported;
      col_bytes += a.row_bytes + a.sbytes[t] + a.zbytes[t];
    }
  }
  a.stage_bytes = cb * col_bytes;
  if (a.stage_bytes * 2 > kRingBudget) return cudaErrorNotSupported;
  a.stages = kRingBudget / a.stage_bytes;
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  a.status = ctx.status;
  int grid = ctx.num_sms;
  if (grid > N) grid = N;
  const int min_grid = (N + kMaxColsPerCta - 1) / kMaxColsPerCta;
  if (grid < min_grid) grid = min_grid;
  const size_t smem = (size_t)a.stages * a.stage_bytes;
  auto kern = select_kernel<PAIR>(wg, cps, bs == 16);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ctx.variant = PAIR ? "gemv_pair_swiglu_tma_ring" : "gemv_tma_ring";
  return launch_kernel(ctx, kern, dim3(grid), dim3(kThreads), smem, a);
}

}  // namespace

cudaError_t launch_gemv_tma(LaunchCtx& ctx, const void* A, const QWeight& w, int K, int N, int bs,
                            void* Y) {
  return launch_tma_impl<false>(ctx, A, &w, K, N, bs, Y);
}

cudaError_t launch_gemv_pair_swiglu_tma(LaunchCtx& ctx, const void* A, const QWeight& gate,
                                        const QWeight& up, int K, int N, int bs, void* out) {
  const QWeight w[2] = {gate, up};
  return launch_tma_impl<true>(ctx, A, w, K, N, bs, out);
}

}  // namespace mnb
