// M = 1 GEMV (and the paired gate/up SwiGLU GEMV) with a bulk-copy (TMA) ring.
//
// A CTA owns a contiguous range of output columns, so its packed weights, scales and
// zero points are three contiguous byte ranges of the MatMulNBits storage.  One producer
// lane streams them, a stage of CB columns at a time, with 1-D `cp.async.bulk` copies
// into a ring of shared-memory slots (up to ~180 KB in flight per SM, independent of the
// register budget).  NCW consumer warps keep their activations in registers, read each
// stage's 16-byte weight chunks from shared memory, form exact fp16 (code - zp) with the
// magic-number conversion, accumulate exact fp16 x fp16 products in fp32, apply the group
// scale to each 32-element partial dot, and reduce per column in a fixed order.
//
// Warps are grouped: WG consumer warps cover one column's K range (lane slot s owns the
// 32-element chunks s, s + 32 WG, ...), and NCW / WG groups work on different columns of
// a stage.  Every wait on an mbarrier is bounded; a wait that gives up records its cause
// in the device status word and the kernel finishes without further shared-memory
// traffic (its outputs are then NaN).
//
// The producer issues its copies before the programmatic-launch wait (the weights are
// never written by the preceding kernel); consumers wait before reading A.
//
// The kernel is specialised on the scale dtype (S16) and on the presence of zero points
// (ZP) so the inner loop carries no per-chunk branches on them; for the paired kernel
// both weights must share those two properties.
#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

constexpr int kMaxColsPerCta = 128;
constexpr int kMaxStages = 8;

struct TmaGemvArgs {
  const __half* A;
  const uint8_t* packed[2];
  const uint8_t* scales[2];
  const uint8_t* zp[2];
  void* Y;
  int K, N, G;
  int group_shift;  // log2(bs / 32) for bs >= 32
  int row_bytes;    // K / 2
  int sbytes;       // scale bytes per row
  int zbytes;       // zero-point bytes per row (0 when absent)
  int stage_bytes;
  int stages;
  uint32_t* status;
  const __half* bias;
  int bias_mode;
  // fp32 activations (AF): A, Y and bias are fp32; Y = acc + bias with no rounding.
  const float* Af;
  float* Yf;
  const float* biasf;
  // Act-order gather (GA): activation k' is A[perm[k']] (0 where perm = -1), A of Ka halves.
  const int32_t* perm;
  int Ka;
  // Zero points read from global memory (ZG): rows of zrb_g bytes that are not 16-byte
  // multiples cannot be bulk-copied per stage; the stage then has no zero-point region.
  int zrb_g;
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

// fp32 activations: the exact fp16 (code - zp) pairs widen to fp32 and multiply fp32
// activations a8[0..7] (word order: nibble i pairs with a8[i], nibble i + 4 with a8[i + 4]).
__device__ __forceinline__ float dot_word_f32(uint32_t w, uint32_t zlo, uint32_t zhi, const float* a8,
                                              float acc) {
  uint32_t d[4];
  nibbles_to_centered_half2(w, zlo, zhi, d);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = *reinterpret_cast<const __half2*>(&d[i]);
    acc = fmaf(__low2float(h), a8[i], acc);
    acc = fmaf(__high2float(h), a8[i + 4], acc);
  }
  return acc;
}

template <int NCW, int WG, int CPS, int VPG, bool BS16, bool PAIR, bool S16, bool ZP, bool AF = false,
          bool GA = false, bool ZG = false>
__global__ void __launch_bounds__((NCW + 1) * 32, (NCW <= 8 ? 2 : 1))
    gemv_tma_kernel(const TmaGemvArgs p) {
  constexpr int kThreads = (NCW + 1) * 32;
  constexpr int NG = NCW / WG;
  constexpr int CB = NG * VPG;
  constexpr int NWT = PAIR ? 2 : 1;
  constexpr int V = VPG * NWT;
  constexpr int kLog2V = (V == 1) ? 0 : (V == 2) ? 1 : (V == 4) ? 2 : (V == 8) ? 3 : 4;
  constexpr int kSB = S16 ? 2 : 4;  // bytes per scale
  static_assert(NG * WG == NCW, "consumer warps must split into whole groups");
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
  const int reg_p = CB * p.row_bytes, reg_s = CB * p.sbytes, reg_z = CB * p.zbytes;
  const int wt_stride = reg_p + reg_s + reg_z;

  if (tid == 0) {
    failed = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ------------------------------- producer -------------------------------------
    if (lane == 0) {
      int issued = 0, slot = 0;
      uint32_t phase = 0;
      for (int st = 0; st < nstages_total; ++st) {
        if (st >= S && !mbar_wait_bounded(&empty_bar[slot], phase ^ 1u)) {
          report_status(p.status, kStatusEmptyWait);
          atomicExch(&failed, 1);
          break;
        }
        const int col = n0 + st * CB;
        const int nc = min(CB, n1 - col);
        const uint32_t bytes = (uint32_t)(nc * NWT) * (p.row_bytes + p.sbytes + p.zbytes);
        uint8_t* base = ring + (size_t)slot * p.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], bytes);
#pragma unroll
        for (int t = 0; t < NWT; ++t) {
          uint8_t* wb = base + t * wt_stride;
          bulk_g2s(wb, p.packed[t] + (long long)col * p.row_bytes, nc * p.row_bytes, &full_bar[slot]);
          bulk_g2s(wb + reg_p, p.scales[t] + (long long)col * p.sbytes, nc * p.sbytes, &full_bar[slot]);
          if (ZP && !ZG)
            bulk_g2s(wb + reg_p + reg_s, p.zp[t] + (long long)col * p.zbytes, nc * p.zbytes,
                     &full_bar[slot]);
        }
        issued = st + 1;
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // Every copy this lane issued must land before the CTA can exit.  Consumers have
      // normally waited for all of them already; after a failed wait this bounds the drain.
      for (int st = issued > S ? issued - S : 0; st < issued; ++st)
        (void)mbar_wait_bounded(&full_bar[st % S], (uint32_t)(st / S) & 1u);
    }
    pdl_launch_dependents();
  } else {
    // ------------------------------- consumers ------------------------------------
    pdl_launch_dependents();
    const int g = warp / WG, wig = warp % WG;
    const int ls = wig * 32 + lane;
    // Act-order gather: consumer thread i places A'[k'] = A[perm[k']] for k' = i, i + 512,
    // ... (at most kGaPer of them).  perm is constant for the weight, so its entries are
    // loaded before the wait; A only after it.
    constexpr int kGaPer = 8192 / (NCW * 32);
    int pidx[GA ? kGaPer : 1];
    if constexpr (GA) {
      static_assert(CPS == 1, "the gathering GEMV keeps one chunk per lane");
#pragma unroll
      for (int u = 0; u < kGaPer; ++u) {
        const int kp = tid + u * NCW * 32;
        pidx[u] = kp < p.K ? __ldg(p.perm + kp) : -1;
      }
    }
    pdl_wait();
    // Act-order gather, in shared memory behind the ring: copy A (Ka halves) with 16-byte
    // loads, permute it into A' (K' halves), then every lane loads its chunk of A' as usual.
    const uint32_t a_u32 = smem_u32(ring) + (uint32_t)(p.stages * p.stage_bytes);
    const uint32_t a2_u32 = a_u32 + (uint32_t)(((p.Ka * 2 + 15) >> 4) << 4);
    if constexpr (GA) {
      for (int i = tid; i < (p.Ka >> 3); i += NCW * 32) {
        const uint4 v = *reinterpret_cast<const uint4*>(p.A + 8 * i);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a_u32 + 16u * (uint32_t)i), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
      bool bad = false;
#pragma unroll
      for (int u = 0; u < kGaPer; ++u) {
        const int kp = tid + u * NCW * 32;
        if (kp < p.K) {
          const int src = pidx[u];
          uint32_t h = 0u;
          if (src >= 0 && src < p.Ka) {
            h = lds_u16_a(a_u32 + 2u * (uint32_t)src);
          } else if (src != -1) {
            bad = true;
          }
          asm volatile("st.shared.u16 [%0], %1;" ::"r"(a2_u32 + 2u * (uint32_t)kp), "h"((unsigned short)h)
                       : "memory");
        }
      }
      if (bad) report_status(p.status, kStatusBadIndex);
      asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
    }

    // Per owned chunk: activations (paired) and byte offsets, inside one column's
    // regions, of its weights, its (first) scale and its zero-point byte.
    uint32_t a[CPS][16];
    float af[AF ? CPS : 1][AF ? 32 : 1];
    uint32_t wofs[CPS], sofs[CPS], zofs[CPS], zsh[CPS];
    bool cval[CPS];
#pragma unroll
    for (int j = 0; j < CPS; ++j) {
      const int c = ls + j * WG * 32;
      cval[j] = c < C;
      wofs[j] = (uint32_t)c * 16u;
      const int gi = BS16 ? 2 * c : (c >> p.group_shift);
      sofs[j] = (uint32_t)gi * kSB;
      zofs[j] = BS16 ? (uint32_t)c : (uint32_t)(gi >> 1);
      zsh[j] = BS16 ? 0u : (uint32_t)((gi & 1) * 4);
      if constexpr (AF) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (cval[j]) x = *reinterpret_cast<const float4*>(p.Af + (long long)c * 32 + q * 4);
          af[j][4 * q] = x.x;
          af[j][4 * q + 1] = x.y;
          af[j][4 * q + 2] = x.z;
          af[j][4 * q + 3] = x.w;
        }
      } else if constexpr (GA) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 x = make_uint4(0, 0, 0, 0);
          if (cval[j]) x = lds128_a(a2_u32 + (uint32_t)c * 64u + (uint32_t)q * 16u);
          pair_halves_stride4(x, &a[j][q * 4]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 x = make_uint4(0, 0, 0, 0);
          if (cval[j]) x = *reinterpret_cast<const uint4*>(p.A + (long long)c * 32 + q * 8);
          pair_halves_stride4(x, &a[j][q * 4]);
        }
      }
    }
    const uint32_t zl8 = zp_lo_const(8u), zh8 = zp_hi_const(8u);
    const uint32_t ring_u32 = smem_u32(ring);

    bool ok = true;
    int slot = 0;
    uint32_t phase = 0;
    for (int st = 0; st < nstages_total; ++st) {
      const int col0 = n0 + st * CB;
      const int nc = min(CB, n1 - col0);
      // ZG: this stage's zero-point bytes, loaded before its wait so the latency overlaps it.
      uint32_t zg[ZG ? VPG : 1][ZG ? CPS : 1];
      if constexpr (ZG) {
#pragma unroll
        for (int vi = 0; vi < VPG; ++vi) {
          const int ci = g + vi * NG;
#pragma unroll
          for (int j = 0; j < CPS; ++j)
            zg[vi][j] = (ci < nc && cval[j]) ? ld_nc_u8(p.zp[0] + (long long)(col0 + ci) * p.zrb_g + zofs[j]) : 0x88u;
        }
      }
      if (ok && !mbar_wait_bounded(&full_bar[slot], phase)) {
        report_status(p.status, kStatusFullWait);
        atomicExch(&failed, 1);
        ok = false;
      }
      const uint32_t sb = ring_u32 + (uint32_t)(slot * p.stage_bytes);
      float part[V];
#pragma unroll
      for (int vi = 0; vi < VPG; ++vi) {
        const int ci = g + vi * NG;
        const bool live = ok && ci < nc;
#pragma unroll
        for (int t = 0; t < NWT; ++t) {
          float acc = 0.0f;
          const uint32_t cp = sb + (uint32_t)(t * wt_stride + ci * p.row_bytes);
          const uint32_t cs = sb + (uint32_t)(t * wt_stride + reg_p + ci * p.sbytes);
          const uint32_t cz = sb + (uint32_t)(t * wt_stride + reg_p + reg_s + ci * p.zbytes);
#pragma unroll
          for (int j = 0; j < CPS; ++j) {
            if (live && cval[j]) {
              const uint4 w4 = lds128_a(cp + wofs[j]);
              uint32_t zb = 0x88u;
              if constexpr (ZG) zb = zg[vi][j];
              else if constexpr (ZP) zb = lds_u8_a(cz + zofs[j]);
              if (BS16) {
                const uint32_t z0 = zb & 15u, z1 = zb >> 4;
                const uint32_t zl0 = ZP ? zp_lo_const(z0) : zl8, zh0 = ZP ? zp_hi_const(z0) : zh8;
                const uint32_t zl1 = ZP ? zp_lo_const(z1) : zl8, zh1 = ZP ? zp_hi_const(z1) : zh8;
                float p0, p1;
                if constexpr (AF) {
                  p0 = dot_word_f32(w4.x, zl0, zh0, &af[j][0], 0.0f);
                  p0 = dot_word_f32(w4.y, zl0, zh0, &af[j][8], p0);
                  p1 = dot_word_f32(w4.z, zl1, zh1, &af[j][16], 0.0f);
                  p1 = dot_word_f32(w4.w, zl1, zh1, &af[j][24], p1);
                } else {
                  p0 = dot_word_tma(w4.x, zl0, zh0, &a[j][0], 0.0f);
                  p0 = dot_word_tma(w4.y, zl0, zh0, &a[j][4], p0);
                  p1 = dot_word_tma(w4.z, zl1, zh1, &a[j][8], 0.0f);
                  p1 = dot_word_tma(w4.w, zl1, zh1, &a[j][12], p1);
                }
                float s0, s1;
                if (S16) {
                  const uint32_t sh = lds_u32_a(cs + sofs[j]);
                  s0 = half_bits_to_float(sh & 0xffffu);
                  s1 = half_bits_to_float(sh >> 16);
                } else {
                  const uint2 sf = lds_u64_a(cs + sofs[j]);
                  s0 = __uint_as_float(sf.x);
                  s1 = __uint_as_float(sf.y);
                }
                acc = fmaf(p0, s0, acc);
                acc = fmaf(p1, s1, acc);
              } else {
                const uint32_t zz = (zb >> zsh[j]) & 15u;
                const uint32_t zlo = ZP ? zp_lo_const(zz) : zl8, zhi = ZP ? zp_hi_const(zz) : zh8;
                float q0, q1;
                if constexpr (AF) {
                  q0 = dot_word_f32(w4.x, zlo, zhi, &af[j][0], 0.0f);
                  q1 = dot_word_f32(w4.y, zlo, zhi, &af[j][8], 0.0f);
                  q0 = dot_word_f32(w4.z, zlo, zhi, &af[j][16], q0);
                  q1 = dot_word_f32(w4.w, zlo, zhi, &af[j][24], q1);
                } else {
                  q0 = dot_word_tma(w4.x, zlo, zhi, &a[j][0], 0.0f);
                  q1 = dot_word_tma(w4.y, zlo, zhi, &a[j][4], 0.0f);
                  q0 = dot_word_tma(w4.z, zlo, zhi, &a[j][8], q0);
                  q1 = dot_word_tma(w4.w, zlo, zhi, &a[j][12], q1);
                }
                const float s = S16 ? half_bits_to_float(lds_u16_a(cs + sofs[j]))
                                    : __uint_as_float(lds_u32_a(cs + sofs[j]));
                acc = fmaf(q0 + q1, s, acc);
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
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
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
    if constexpr (AF) {
      float out = v[0] + (p.biasf ? p.biasf[n0 + c] : 0.0f);
      if (bad) out = __uint_as_float(0x7fc00000u);
      p.Yf[n0 + c] = out;
    } else {
      __half out;
      if (PAIR) out = __float2half_rn(silu_f32(v[0]) * v[NWT - 1]);
      else out = round_out(v[0], p.bias, n0 + c, p.bias_mode);
      if (bad) out = __ushort_as_half(0x7e00);
      reinterpret_cast<__half*>(p.Y)[n0 + c] = out;
    }
  }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
// Sixteen consumer warps per CTA and one CTA per SM: enough warps per scheduler to keep
// the conversion and FMA pipes issuing while the ring streams.
constexpr int kNCW = 16;
constexpr int kRingBudget = 180 * 1024;
// The paired kernel's stages hold twice the bytes; three of them need a larger ring (a
// larger ring did not help the single-weight kernel).
constexpr int kRingBudgetPair = 210 * 1024;

using TmaKernel = void (*)(const TmaGemvArgs);

template <int WG, int CPS, bool PAIR>
TmaKernel pick(bool bs16, bool s16, bool zp) {
  // Columns per lane group and stage: four; two for the pair beyond one chunk per lane,
  // whose stages would not fit the ring otherwise.
  constexpr int VPG = (PAIR && CPS > 1) ? 2 : 4;
#define MNB_PICK(B, S, Z) gemv_tma_kernel<kNCW, WG, CPS, VPG, B, PAIR, S, Z>
  if (bs16) {
    if (s16) return zp ? MNB_PICK(true, true, true) : MNB_PICK(true, true, false);
    return zp ? MNB_PICK(true, false, true) : MNB_PICK(true, false, false);
  }
  if (s16) return zp ? MNB_PICK(false, true, true) : MNB_PICK(false, true, false);
  return zp ? MNB_PICK(false, false, true) : MNB_PICK(false, false, false);
#undef MNB_PICK
}

// fp32 activations (single weight, at most two chunks per lane so the fp32 activations
// stay in registers).
template <int WG, int CPS>
TmaKernel pick_af(bool bs16, bool s16, bool zp) {
#define MNB_PICK(B, S, Z) gemv_tma_kernel<kNCW, WG, CPS, 4, B, false, S, Z, true>
  if (bs16) {
    if (s16) return zp ? MNB_PICK(true, true, true) : MNB_PICK(true, true, false);
    return zp ? MNB_PICK(true, false, true) : MNB_PICK(true, false, false);
  }
  if (s16) return zp ? MNB_PICK(false, true, true) : MNB_PICK(false, true, false);
  return zp ? MNB_PICK(false, false, true) : MNB_PICK(false, false, false);
#undef MNB_PICK
}

// Zero points from global memory (single weight, fp16 activations).
template <int WG, int CPS>
TmaKernel pick_zg(bool bs16, bool s16) {
#define MNB_PICK(B, S) gemv_tma_kernel<kNCW, WG, CPS, 4, B, false, S, true, false, false, true>
  if (bs16) return s16 ? MNB_PICK(true, true) : MNB_PICK(true, false);
  return s16 ? MNB_PICK(false, true) : MNB_PICK(false, false);
#undef MNB_PICK
}

// Act-order gather (single weight, one chunk per lane).
template <int WG>
TmaKernel pick_ga(bool bs16, bool s16, bool zp) {
#define MNB_PICK(B, S, Z) gemv_tma_kernel<kNCW, WG, 1, 4, B, false, S, Z, false, true>
  if (bs16) {
    if (s16) return zp ? MNB_PICK(true, true, true) : MNB_PICK(true, true, false);
    return zp ? MNB_PICK(true, false, true) : MNB_PICK(true, false, false);
  }
  if (s16) return zp ? MNB_PICK(false, true, true) : MNB_PICK(false, true, false);
  return zp ? MNB_PICK(false, false, true) : MNB_PICK(false, false, false);
#undef MNB_PICK
}

template <bool PAIR>
TmaKernel select_kernel(int wg, int cps, bool bs16, bool s16, bool zp, bool af, bool ga, bool zgl) {
  if (zgl) {
    if (wg == 4) return pick_zg<4, 1>(bs16, s16);
    return cps == 1 ? pick_zg<8, 1>(bs16, s16) : pick_zg<8, 2>(bs16, s16);
  }
  if (ga) return wg == 4 ? pick_ga<4>(bs16, s16, zp) : pick_ga<8>(bs16, s16, zp);
  if (af) {
    if (wg == 4) return pick_af<4, 1>(bs16, s16, zp);
    if (cps == 1) return pick_af<8, 1>(bs16, s16, zp);
    return pick_af<8, 2>(bs16, s16, zp);
  }
  if (wg == 4) return pick<4, 1, PAIR>(bs16, s16, zp);
  if (cps == 1) return pick<8, 1, PAIR>(bs16, s16, zp);
  if (cps == 2) return pick<8, 2, PAIR>(bs16, s16, zp);
  return pick<8, 4, PAIR>(bs16, s16, zp);
}

template <bool PAIR>
cudaError_t launch_tma_impl(LaunchCtx& ctx, const void* A, const QWeight* w, int K, int N, int bs,
                            void* Y, const float* Af = nullptr, float* Yf = nullptr,
                            const float* biasf = nullptr, const int32_t* perm = nullptr, int Ka = 0) {
  constexpr int NWT = PAIR ? 2 : 1;
  const bool af = Af != nullptr;
  const bool ga = perm != nullptr;
  if (K % 32 != 0) return cudaErrorNotSupported;
  if (PAIR && (w[0].scales_f16 != w[1].scales_f16 || (w[0].zp == nullptr) != (w[1].zp == nullptr)))
    return cudaErrorNotSupported;
  const int C = K / 32;
  // Four warps cover K <= 4096 (one chunk per lane); eight warps with one, two or four
  // chunks per lane cover K <= 32768.
  int wg, cps;
  if (C <= 128) {
    wg = 4;
    cps = 1;
  } else {
    wg = 8;
    cps = (C + 255) / 256;
    if (cps == 3) cps = 4;
    if (cps > 4 || (af && cps > 2)) return cudaErrorNotSupported;
  }
  if (ga && cps != 1) return cudaErrorNotSupported;
  const int ng = kNCW / wg;
  const int cb = ng * ((PAIR && cps > 1) ? 2 : 4);
  const int G = K / bs;
  const bool s16 = w[0].scales_f16 != 0;
  const bool zp = w[0].zp != nullptr;
  TmaGemvArgs a = {};
  a.A = static_cast<const __half*>(A);
  a.Y = Y;
  a.K = K;
  a.N = N;
  a.G = G;
  a.row_bytes = K / 2;
  a.group_shift = 0;
  while (bs >= 32 && (32 << a.group_shift) < bs) ++a.group_shift;
  a.sbytes = G * (s16 ? 2 : 4);
  a.zbytes = zp ? (G + 1) / 2 : 0;
  a.zrb_g = a.zbytes;
  // Zero-point rows that are not 16-byte multiples: read from global memory instead of
  // staged (single fp16-activation weight only).
  const bool zgl = zp && a.zbytes % 16 != 0 && !PAIR && !af && !ga;
  if (zgl) {
    if (cps > 2) return cudaErrorNotSupported;  // keeps the per-stage zero points in registers
    a.zbytes = 0;
  }
  if (a.sbytes % 16 != 0 || a.zbytes % 16 != 0) return cudaErrorNotSupported;
  for (int t = 0; t < 2; ++t) {
    const QWeight& q = w[t < NWT ? t : 0];
    a.packed[t] = q.packed;
    a.scales[t] = static_cast<const uint8_t*>(q.scales);
    a.zp[t] = q.zp;
  }
  a.stage_bytes = cb * NWT * (a.row_bytes + a.sbytes + a.zbytes);
  // Shared copies of A and of the permuted A' for the gather.
  const int abytes = ga ? (Ka * 2 + 15) / 16 * 16 + K * 2 : 0;
  const int ring_budget = (PAIR ? kRingBudgetPair : kRingBudget) - abytes;
  if (a.stage_bytes * 2 > ring_budget) return cudaErrorNotSupported;
  a.stages = ring_budget / a.stage_bytes;
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  a.status = ctx.status;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = PAIR ? 0 : ctx.bias_mode;
  a.Af = Af;
  a.Yf = Yf;
  a.biasf = biasf;
  a.perm = perm;
  a.Ka = Ka;
  int grid = ctx.num_sms;
  if (grid > N) grid = N;
  const int min_grid = (N + kMaxColsPerCta - 1) / kMaxColsPerCta;
  if (grid < min_grid) grid = min_grid;
  const size_t smem = (size_t)a.stages * a.stage_bytes + abytes;
  auto kern = select_kernel<PAIR>(wg, cps, bs == 16, s16, zp, af, ga, zgl);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ctx.variant = PAIR ? "gemv_pair_swiglu_tma_ring"
                     : (af ? "gemv_f32_tma_ring" : (ga ? "gemv_tma_ring_gather" : "gemv_tma_ring"));
  return launch_kernel(ctx, kern, dim3(grid), dim3((kNCW + 1) * 32), smem, a);
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

cudaError_t launch_gemv_f32_tma(LaunchCtx& ctx, const float* A, const QWeight& w, int K, int N, int bs,
                                float* Y, const float* bias) {
  return launch_tma_impl<false>(ctx, nullptr, &w, K, N, bs, nullptr, A, Y, bias);
}

cudaError_t launch_gemv_tma_gather(LaunchCtx& ctx, const void* A, const int32_t* perm, int Ka, const QWeight& w,
                                   int Kp, int N, int bs, void* Y) {
  return launch_tma_impl<false>(ctx, A, &w, Kp, N, bs, Y, nullptr, nullptr, nullptr, perm, Ka);
}

}  // namespace mnb
