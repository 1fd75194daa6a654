// M > 16 GEMM on the tcgen05 tensor cores: Y[M,N] = A[M,K] . dequant(B)^T.
//
// Orientation: the dequantised weights are the MMA's A operand (M_mma = 128 weight rows,
// i.e. 128 output columns n) and the activations are its B operand (N_mma = 256 rows m),
// so the accumulator tile D[n, m] sits in TMEM with one weight row per TMEM lane.  The
// per-group scale of row n is then a per-thread scalar in the epilogue, and "scale after
// accumulate" (marlin_gemm.rs: per-group scaling applied after the tensor-core
// accumulate) costs one FMA per accumulator element per group.
//
// Roles in a 512-thread CTA (one persistent CTA per SM, tiles of 128 n x 256 m):
//   warp 0      producer: per 64-k stage, a 2-D TMA load of the 256 x 64 activation box
//               (128-byte swizzle) and a 1-D bulk copy of the 4 KB repacked weight block
//               into a 4-deep ring (36 KB a slot);
//   warp 1      MMA issuer (one lane) and TMEM owner (512 columns: two 256-column
//               partial accumulators, one per quant group in flight);
//   warps 4-7   dequantisers: repacked nibbles -> exact fp16 (code - zp) written into one of
//               four 16 KB weight buffers in the K-major 128-byte-swizzled operand layout
//               (four, so the dequantisers run up to three stages ahead of the MMAs);
//   warps 8-15  epilogue: per group, read the partial from TMEM, multiply by the group
//               scale, add into fp32 registers; at the end of a tile, store fp16 Y.
// Register split (setmaxnreg, warpgroup granularity, launch = 512 x 128):
//   warpgroup 0: 64, warpgroup 1: 80, warpgroups 2-3: 184 -> 128 x (64+80+184+184) = 65536.
// Every mbarrier wait is bounded; a wait that gives up sets the device status word and
// the role stops, so the kernel always terminates.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mnb_device.cuh"
#include "mnb_internal.h"
#include "tcgen05.cuh"

namespace mnb {
namespace {

constexpr int kTileN = 128;  // weight rows per tile (M_mma)
constexpr int kTileM = 256;  // activation rows per tile (N_mma)
constexpr int kStageK = 64;
constexpr int kStages = 4;                       // activation + packed-weight ring
constexpr int kWBufs = 4;                        // dequantised-weight buffers (<= kStages)
constexpr int kXBytes = kTileM * kStageK * 2;   // 32 KB
constexpr int kPBytes = kTileN * kStageK / 2;   // 4 KB
constexpr int kWBytes = kTileN * kStageK * 2;   // 16 KB
constexpr int kStageBytes = kXBytes + kPBytes;   // one ring slot (1024-aligned)
constexpr int kWOffset = kStages * kStageBytes;  // start of the weight buffers
constexpr int kSmemBytes = kWOffset + kWBufs * kWBytes + 1024;
constexpr int kThreads = 512;
constexpr uint32_t kTmemCols = 512;

struct TcArgs {
  const uint8_t* repacked;
  const uint8_t* scales;
  const uint8_t* zp;
  int scales_f16;
  __half* Y;
  int M, N, K, bs, G, zrb;
  int kblocks;  // ceil(K / 64)
  int nmma;     // MMA N = activation rows per tile: 256, or M rounded up to 16 when M < 256
                // (one tile row; accumulator columns past it are never written nor stored)
  int mtiles, ntiles;
  uint32_t* status;
  const __half* bias;
  int bias_mode;
  // fp32 output (F32): the activation operand has 2 * Mout rows, row 2m = hi and row
  // 2m + 1 = lo of fp32 row m scaled by 2^-rexp[m]; the two accumulator columns of a
  // pair sit next to each other in one epilogue thread, which stores
  // Yf[m, n] = 2^rexp[m] * (acc[2m] + acc[2m + 1]) + biasf[n].
  int Mout;
  float* Yf;
  const float* biasf;
  const int* rexp;
  // Split-K (few output tiles): work item t is slice t % ksplit of tile t / ksplit, a range
  // of whole quant groups (kunit k-blocks each); every item stores its fp32 partial
  // part[slice][m][n] (rows of the activation operand), summed afterwards in slice order.
  int ksplit, kunit;
  float* part;
};

// k-block range [lo, hi) of slice `sl` (whole units of p.kunit k-blocks).
__device__ __forceinline__ void slice_range(const TcArgs& p, int sl, int& lo, int& hi) {
  const int nunits = p.kblocks / p.kunit;
  lo = (sl * nunits / p.ksplit) * p.kunit;
  hi = ((sl + 1) * nunits / p.ksplit) * p.kunit;
}

__device__ __forceinline__ uint32_t zp_byte(const TcArgs& p, int n, int byte_idx) {
  if (p.zp == nullptr || n >= p.N || byte_idx >= p.zrb) return 0x88u;
  return ld_nc_u8(p.zp + (long long)n * p.zrb + byte_idx);
}

template <bool F32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const TcArgs p, const __grid_constant__ CUtensorMap tmap_a) {
  const int ksplit = p.ksplit;  // K slices per tile (1: unsplit)
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint64_t wready_bar[kWBufs];
  __shared__ uint64_t tfull_bar[2], tempty_bar[2], mma_done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int KS = p.K / 16;                   // MMA k-steps per tile
  const int ntile_total = p.mtiles * p.ntiles * ksplit;  // work items

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < kWBufs; ++s) mbar_init(&wready_bar[s], 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 8);
    }
    mbar_init(&mma_done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  auto stage_x = [&](int s) { return smem + s * kStageBytes; };
  auto stage_p = [&](int s) { return smem + s * kStageBytes + kXBytes; };

  const int wg = warp >> 2;
  if (wg == 0) {
    tc::setmaxnreg_dec<64>();
    if (warp == 0 && lane == 0) {
      // ------------------------------ producer ------------------------------------
      tc::prefetch_tmap(&tmap_a);
      pdl_launch_dependents();
      pdl_wait();  // the activations may come from the previous kernel
      int slot = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntile_total && ok; t += gridDim.x) {
        const int tile = t / ksplit;
        const int mt = tile % p.mtiles, nt = tile / p.mtiles;
        int kb_lo, kb_hi;
        slice_range(p, t % ksplit, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (issued >= kStages && !mbar_wait_bounded(&empty_bar[slot], phase ^ 1u)) {
            report_status(p.status, kStatusEmptyWait);
            atomicExch(&abort_flag, 1);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(p.nmma * kStageK * 2 + kPBytes));
          tc::tma_load_2d(stage_x(slot), &tmap_a, kb * kStageK, mt * kTileM, &full_bar[slot]);
          bulk_g2s(stage_p(slot), p.repacked + ((long long)nt * p.kblocks + kb) * kPBytes, kPBytes,
                   &full_bar[slot]);
          ++issued;
          if (++slot == kStages) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every copy land before the CTA can retire.
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        (void)mbar_wait_bounded(&full_bar[i % kStages], (uint32_t)(i / kStages) & 1u);
    } else if (warp == 1 && lane == 0) {
      // ------------------------------ MMA issuer ----------------------------------
      // The tensor pipe queues about one MMA, so any work between two tcgen05.mma idles
      // it: the four descriptors of a stage are formed before its first MMA, group
      // boundaries are precomputed, and waits spin without suspending.
      pdl_launch_dependents();
      const uint32_t idesc = tc::idesc_f16_f32(kTileN, p.nmma);
      const uint64_t dx0 = tc::smem_desc_k_sw128(smem_u32(smem));
      const uint64_t dw0 = tc::smem_desc_k_sw128(smem_u32(smem) + kWOffset);
      const uint32_t kpg_mask = (uint32_t)(p.bs / 16) - 1u;  // k-steps per group - 1
      uint32_t slot = 0, phase = 0, b = 0, gphase = 0, wb = 0, wphase = 0;
      uint32_t ngroups = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntile_total && ok; t += gridDim.x) {
        int kb_lo, kb_hi;
        slice_range(p, t % ksplit, kb_lo, kb_hi);
        uint32_t ks = (uint32_t)kb_lo * 4u;  // absolute k-step (group boundaries)
        for (int kb = kb_lo; kb < kb_hi && ok; ++kb) {
          // The dequantisers arrive on wready only after observing this stage's full
          // barrier (which also covers the activation box), so one wait orders both.
          if (!mbar_spin_bounded(&wready_bar[wb], wphase)) {
            report_status(p.status, kStatusMmaWait);
            atomicExch(&abort_flag, 1);
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t ax = dx0 + (uint64_t)((slot * (uint32_t)kStageBytes) >> 4);
          const uint64_t aw = dw0 + (uint64_t)((wb * (uint32_t)kWBytes) >> 4);
          const uint32_t nk = min(4u, (uint32_t)KS - ks);
          if (nk == 4u && kpg_mask >= 3u) {
            // Whole stage inside one group (bs >= 64): at most one group start (first
            // k-step) and one group end (last k-step).
            const bool starts = (ks & kpg_mask) == 0u;
            const bool ends = ((ks + 3u) & kpg_mask) == kpg_mask;
            if (starts && ngroups >= 2u) {
              if (!mbar_spin_bounded(&tempty_bar[b], gphase ^ 1u)) {
                report_status(p.status, kStatusMmaWait);
                atomicExch(&abort_flag, 1);
                ok = false;
                break;
              }
              tc::fence_after_sync();
            }
            const uint32_t d = tmem + b * 256u;
            tc::mma_f16(d, aw, ax, idesc, starts ? 0u : 1u);
            tc::mma_f16(d, aw + 2u, ax + 2u, idesc, 1u);
            tc::mma_f16(d, aw + 4u, ax + 4u, idesc, 1u);
            tc::mma_f16(d, aw + 6u, ax + 6u, idesc, 1u);
            ks += 4u;
            tc::mma_commit(&empty_bar[slot]);  // ring slot and weight buffer free
            if (ends) {
              tc::mma_commit(&tfull_bar[b]);
              ++ngroups;
              b ^= 1u;
              if (b == 0u) gphase ^= 1u;
            }
          } else {
            for (uint32_t kk = 0; kk < nk; ++kk) {
              const bool first = (ks & kpg_mask) == 0u;
              if (first && ngroups >= 2u) {
                if (!mbar_spin_bounded(&tempty_bar[b], gphase ^ 1u)) {
                  report_status(p.status, kStatusMmaWait);
                  atomicExch(&abort_flag, 1);
                  ok = false;
                  break;
                }
                tc::fence_after_sync();
              }
              tc::mma_f16(tmem + b * 256u, aw + 2u * kk, ax + 2u * kk, idesc, first ? 0u : 1u);
              if ((ks & kpg_mask) == kpg_mask) {  // last k-step of the group
                tc::mma_commit(&tfull_bar[b]);
                ++ngroups;
                b ^= 1u;
                if (b == 0u) gphase ^= 1u;
              }
              ++ks;
            }
            if (!ok) break;
            tc::mma_commit(&empty_bar[slot]);  // ring slot and weight buffer free
          }
          if (++slot == (uint32_t)kStages) {
            slot = 0;
            phase ^= 1u;
          }
          if (++wb == (uint32_t)kWBufs) {
            wb = 0u;
            wphase ^= 1u;
          }
        }
      }
      tc::mma_commit(&mma_done_bar);
      (void)mbar_wait_bounded(&mma_done_bar, 0);
    }
  } else if (wg == 1) {
    tc::setmaxnreg_dec<80>();
    pdl_launch_dependents();
    // ------------------------------ dequantisers -------------------------------------
    const int r = tid - 128;  // weight row within the tile
    int gshift = 0;           // log2(block size)
    while ((1 << gshift) < p.bs) ++gshift;
    int slot = 0, wb = 0, si = 0;
    uint32_t phase = 0;
    int pslot = 0;          // ring slot of stage si - kWBufs
    uint32_t pphase = 0;    // parity of that slot's completed "empty" phase
    bool ok = true;
    const uint32_t w_u32 = smem_u32(smem) + kWOffset;
    for (int t = blockIdx.x; t < ntile_total && ok; t += gridDim.x) {
      const int nt = (t / ksplit) / p.mtiles;
      const int n = nt * kTileN + r;
      int kb_lo, kb_hi;
      slice_range(p, t % ksplit, kb_lo, kb_hi);
      // Zero-point byte(s) covering one 64-k stage: one byte for bs >= 32 (two groups at
      // most, sharing a byte), two bytes for bs = 16.
      auto zp_for = [&](int kb) -> uint32_t {
        const int g0 = (kb * kStageK) >> gshift;
        if (gshift == 4) return zp_byte(p, n, g0 >> 1) | (zp_byte(p, n, (g0 >> 1) + 1) << 8);
        return zp_byte(p, n, g0 >> 1);
      };
      // One stage: wait for its codes and a free weight buffer, convert, store, announce.
      auto do_stage = [&](int kb, uint32_t zcur) -> bool {
        // The weight buffer was last read by stage si - kWBufs, whose completion is that
        // stage's ring-slot "empty" phase.
        if (!mbar_wait_bounded(&full_bar[slot], phase) ||
            (si >= kWBufs && !mbar_wait_bounded(&empty_bar[pslot], pphase)))
          return false;
        const uint8_t* sp = stage_p(slot);
        const uint32_t sw = w_u32 + (uint32_t)(wb * kWBytes) + (uint32_t)(r * 128);
        const int g0 = (kb * kStageK) >> gshift;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 v = lds128(sp + q * 2048 + r * 16);
          const uint32_t words[4] = {v.x, v.y, v.z, v.w};
          // zero points of this 32-k half: one group for bs >= 32, two for bs = 16
          const int gq = (kb * kStageK + q * 32) >> gshift;
          uint32_t za, zb2;
          if (gshift == 4) {
            za = (zcur >> ((gq - g0) * 4)) & 15u;
            zb2 = (zcur >> ((gq + 1 - g0) * 4)) & 15u;
          } else {
            za = (gq & 1) ? ((zcur >> 4) & 15u) : (zcur & 15u);
            zb2 = za;
          }
          const uint32_t zla = zp_lo_const(za), zha = zp_hi_const(za);
          const uint32_t zlb = zp_lo_const(zb2), zhb = zp_hi_const(zb2);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t d[4];
            nibbles_to_centered_half2(words[j], j < 2 ? zla : zlb, j < 2 ? zha : zhb, d);
            const int c = q * 4 + j;  // 16-byte chunk (8 k) within the 128-byte row
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(sw + (uint32_t)((c ^ (r & 7)) << 4)),
                         "r"(d[0]), "r"(d[1]), "r"(d[2]), "r"(d[3])
                         : "memory");
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&wready_bar[wb]);
        if (++slot == kStages) {
          slot = 0;
          phase ^= 1u;
        }
        if (++wb == kWBufs) wb = 0;
        if (si >= kWBufs) {  // advance the (si - kWBufs) cursor once it has been used
          if (++pslot == kStages) {
            pslot = 0;
            pphase ^= 1u;
          }
        }
        ++si;
        return true;
      };
      // Two zero-point registers, one per stage parity, each reloaded two stages ahead right
      // after its last use, so no register copy ever waits for a global load in flight.
      uint32_t zeven = zp_for(kb_lo);
      uint32_t zodd = kb_lo + 1 < kb_hi ? zp_for(kb_lo + 1) : 0u;
      for (int kb = kb_lo; kb < kb_hi && ok; kb += 2) {
        if (!do_stage(kb, zeven)) {
          ok = false;
          break;
        }
        if (kb + 2 < kb_hi) zeven = zp_for(kb + 2);
        if (kb + 1 < kb_hi) {
          if (!do_stage(kb + 1, zodd)) {
            ok = false;
            break;
          }
          if (kb + 3 < kb_hi) zodd = zp_for(kb + 3);
        }
      }
      if (!ok) {
        report_status(p.status, kStatusFullWait);
        atomicExch(&abort_flag, 1);
      }
    }
  } else {
    tc::setmaxnreg_inc<184>();
    pdl_launch_dependents();
    // ------------------------------ epilogue ----------------------------------------
    const int e = warp - 8;          // 0..7
    const int quarter = warp & 3;    // TMEM lanes 32*quarter .. +31
    const int half = e >> 2;         // columns 128*half .. +127
    long long gc = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntile_total && ok; t += gridDim.x) {
      const int tile = t / ksplit, sl = t % ksplit;
      const int mt = tile % p.mtiles, nt = tile / p.mtiles;
      const int n = nt * kTileN + quarter * 32 + lane;
      const bool nval = n < p.N;
      int kb_lo, kb_hi;
      slice_range(p, sl, kb_lo, kb_hi);
      const int g_lo = (kb_lo * kStageK) / p.bs;
      const int g_hi = ksplit > 1 ? (kb_hi * kStageK) / p.bs : p.G;
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
      auto scale_of = [&](int g) -> float {
        if (!nval) return 0.0f;
        const long long si = (long long)n * p.G + g;
        return p.scales_f16 ? half_bits_to_float(ld_nc_u16(p.scales + 2 * si))
                            : __uint_as_float(ld_nc_u32(p.scales + 4 * si));
      };
      float s_next = scale_of(g_lo);
      for (int g = g_lo; g < g_hi; ++g) {
        const float s = s_next;
        if (g + 1 < g_hi) s_next = scale_of(g + 1);
        const uint32_t b = (uint32_t)(gc & 1);
        if (!mbar_wait_bounded(&tfull_bar[b], (uint32_t)((gc >> 1) & 1))) {
          report_status(p.status, kStatusMmaWait);
          atomicExch(&abort_flag, 1);
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t tbase = tmem + b * 256u + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          // accumulator columns at or past the MMA's N hold nothing (the condition is the same
          // for the whole warp, as the collective TMEM load requires)
          if (half * 128 + c * 32 < p.nmma) {
            float v[32];
            tc::tmem_ld32(tbase + c * 32, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c * 32 + i] = fmaf(v[i], s, acc[c * 32 + i]);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[b]);
        ++gc;
      }
      if (!ok) break;
      if (ksplit > 1) {
       if (nval) {
        // plain fp32 partial of this slice, every row of the activation operand
        float* pc = p.part + (long long)sl * p.M * p.N + n;
        const int m0 = mt * kTileM + half * 128;
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const int m = m0 + i;
          if (m < p.M) pc[(long long)m * p.N] = acc[i];
        }
       }
      } else if (nval) {
        const int m0 = mt * kTileM + half * 128;
        if constexpr (F32) {
          const float b = p.biasf ? p.biasf[n] : 0.0f;
          float* yc = p.Yf + n;
          const int mo0 = m0 >> 1;  // m0 is even: columns 2i and 2i + 1 are one fp32 row
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const int mo = mo0 + i;
            if (mo < p.Mout) yc[(long long)mo * p.N] = ldexpf(acc[2 * i] + acc[2 * i + 1], p.rexp[mo]) + b;
          }
        } else {
          __half* yc = p.Y + n;
#pragma unroll
          for (int i = 0; i < 128; ++i) {
            const int m = m0 + i;
            if (m < p.M) yc[(long long)m * p.N] = round_out(acc[i], p.bias, n, p.bias_mode);
          }
        }
      }
    }
    if (abort_flag) {
      // A wait gave up somewhere: mark this CTA's outputs as invalid.
      for (int t = blockIdx.x; t < ntile_total; t += gridDim.x) {
        const int tile = t / ksplit;
        const int mt = tile % p.mtiles, nt = tile / p.mtiles;
        const int n = nt * kTileN + quarter * 32 + lane;
        if (n >= p.N) continue;
        for (int i = 0; i < 128; ++i) {
          const int m = mt * kTileM + half * 128 + i;
          if (ksplit > 1) {
            if (m < p.M) p.part[((long long)(t % ksplit) * p.M + m) * p.N + n] = __uint_as_float(0x7fc00000u);
          } else if constexpr (F32) {
            if ((m & 1) == 0 && (m >> 1) < p.Mout) p.Yf[(long long)(m >> 1) * p.N + n] = __uint_as_float(0x7fc00000u);
          } else {
            if (m < p.M) p.Y[(long long)m * p.N + n] = __ushort_as_half(0x7e00);
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// ----------------------------------------------------------------------------------
// Host: tensor map for the activations (K innermost), cached driver entry point.
// ----------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

size_t gemm_tc_smem_bytes() { return kSmemBytes; }

void* tensor_map_encode_fn() { return reinterpret_cast<void*>(get_encode()); }

namespace {

// K slices for an M-row (activation operand) x N output on num_sms SMs: 1 unless the
// output has fewer tiles than half the SMs; slices are whole quant groups of at least four
// 64-k blocks, at most 32 of them.
int tc_ksplit(int M, int K, int N, int bs, int num_sms) {
  if (K % kStageK != 0 || K % bs != 0) return 1;
  const int tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
  if (2 * tiles > num_sms) return 1;
  const int kblocks = K / kStageK, unit = bs > kStageK ? bs / kStageK : 1;
  int ks = num_sms / tiles;
  if (ks > kblocks / 4) ks = kblocks / 4;
  if (ks > kblocks / unit) ks = kblocks / unit;
  if (ks > 32) ks = 32;
  return ks < 2 ? 1 : ks;
}

constexpr int kMaxSms = 160;  // workspace sizing covers any GPU with up to this many SMs

cudaError_t launch_tc_impl(LaunchCtx& ctx, const void* A, int M, const QWeight& w, const uint8_t* repacked, int K,
                           int N, int bs, void* Y, int Mout, float* Yf, const float* biasf, const int* rexp,
                           void* workspace, size_t ws_bytes) {
  if (K % 16 != 0) return cudaErrorNotSupported;
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
  const int nmma = M >= kTileM ? kTileM : (M + 15) / 16 * 16;
  const cuuint32_t box[2] = {(cuuint32_t)kStageK, (cuuint32_t)nmma};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(A), gdim, gstride, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  TcArgs a = {};
  a.repacked = repacked;
  a.scales = static_cast<const uint8_t*>(w.scales);
  a.zp = w.zp;
  a.scales_f16 = w.scales_f16;
  a.Y = static_cast<__half*>(Y);
  a.M = M;
  a.N = N;
  a.K = K;
  a.bs = bs;
  a.G = K / bs;
  a.zrb = (a.G + 1) / 2;
  a.kblocks = (K + kStageK - 1) / kStageK;
  a.nmma = nmma;
  a.mtiles = (M + kTileM - 1) / kTileM;
  a.ntiles = (N + kTileN - 1) / kTileN;
  a.status = ctx.status;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = ctx.bias_mode;
  a.Mout = Mout;
  a.Yf = Yf;
  a.biasf = biasf;
  a.rexp = rexp;
  a.ksplit = tc_ksplit(M, K, N, bs, ctx.num_sms);
  if (a.ksplit > 1 && (workspace == nullptr || ws_bytes < (size_t)a.ksplit * M * N * 4)) a.ksplit = 1;
  a.kunit = bs > kStageK ? bs / kStageK : 1;
  a.part = static_cast<float*>(workspace);
  const int items = a.mtiles * a.ntiles * a.ksplit;
  const int grid = items < ctx.num_sms ? items : ctx.num_sms;
  const bool f32 = Yf != nullptr;
  auto kern = f32 ? gemm_tc_kernel<true> : gemm_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_kernel(ctx, kern, dim3(grid), dim3(kThreads), (size_t)kSmemBytes, a, tmap);
  ctx.variant = f32 ? "gemm_tcgen05_w128xa256_f32split" : "gemm_tcgen05_w128xa256";
  if (e != cudaSuccess || a.ksplit == 1) return e;
  ctx.variant = f32 ? "gemm_tcgen05_w128xa256_f32split_splitk" : "gemm_tcgen05_w128xa256_splitk";
  if (f32) return launch_combine_slices_f32(ctx, a.part, a.ksplit, Mout, N, Yf, biasf, rexp);
  return launch_combine_slices(ctx, a.part, a.ksplit, M, N, Y);
}

}  // namespace

size_t gemm_tc_workspace_bytes(int M_rows, int K, int N, int bs) {
  const int ks = tc_ksplit(M_rows, K, N, bs, kMaxSms);
  return ks > 1 ? (size_t)ks * M_rows * N * 4 : 0;
}

cudaError_t launch_gemm_tc(LaunchCtx& ctx, const void* A, int M, const QWeight& w,
                           const uint8_t* repacked, int K, int N, int bs, void* Y, void* workspace, size_t ws_bytes) {
  return launch_tc_impl(ctx, A, M, w, repacked, K, N, bs, Y, M, nullptr, nullptr, nullptr, workspace, ws_bytes);
}

cudaError_t launch_gemm_tc_f32split(LaunchCtx& ctx, const void* A2, int M, const QWeight& w,
                                    const uint8_t* repacked, int K, int N, int bs, float* Y, const float* bias,
                                    const int* rexp, void* workspace, size_t ws_bytes) {
  return launch_tc_impl(ctx, A2, 2 * M, w, repacked, K, N, bs, nullptr, M, Y, bias, rexp, workspace, ws_bytes);
}

}  // namespace mnb
