// M = 1 GEMV (and the paired gate/up SwiGLU GEMV) with the multiply-accumulate on the
// tensor cores: mma.sync m16n8k16, fp16 operands, fp32 accumulate.
//
// Why: a decode GEMV moves ~0.58 bytes per weight, and at HBM rate a CUDA-core inner loop
// (nibble conversion plus one mixed-precision FMA per weight) runs out of instruction
// issue before it runs out of bandwidth.  Here the conversion is the only per-weight work:
// the products and sums go to the tensor cores, ~1.6 issued instructions per weight
// instead of ~3.2.
//
// Data flow.  A CTA owns a contiguous range of 16-row weight tiles (rows are output
// columns n).  A producer warp streams each tile, optionally in K slices, into a ring of
// shared-memory stages: packed rows by one 1-D bulk copy per row at a stride of
// (slice bytes + 16), scales as 128-byte-swizzled 2-D tensor boxes (16 rows x 128 bytes),
// zero points as one copy of the tile's rows.  Consumer warps split each tile's K range
// into blocks of 256 k (8 chunks of 32 k) and walk their blocks in every tile.
//
// The MMA mapping.  Lane (g, t) (g = lane / 4, t = lane % 4) reads the two 16-byte chunks
// 2t and 2t + 1 of a block from rows g and g + 8 and converts each 32-bit word into exact
// fp16 (code - zp) (magic-number conversion, zero point folded into its constants).  Word
// q of chunk 2t feeds the "X" MMAs of step q and word q of chunk 2t + 1 the "Y" MMAs, as
// the A operand (rows g, g + 8; the k order inside an MMA is the conversion's pairing,
// used identically for both operands).  The B operand holds the activation: column c of
// B carries chunk c of the block at the k slots of lane c / 2 and zero elsewhere, so in
// the X MMAs column 2t of D is row n's partial dot with chunk 2t, and in the Y MMAs column
// 2t + 1 is its partial dot with chunk 2t + 1; the other columns are never read.  Lane
// (g, t) therefore receives exactly the partial dots of its own chunks (D registers 0 and
// 2 of X, 1 and 3 of Y) and multiplies each by the scale of its group (scale after the
// partial dot of each 32-element chunk, as the fp16 GEMV of matmul_nbits.rs applies its
// per-block scale), accumulating in fp32.  Only 8 lanes of a warp load B; the other lanes
// keep zero registers.
//
// Bank conflicts.  Packed rows sit at a stride of 16 mod 128 bytes, so the 8 lanes of a
// quarter-warp (rows g, g + 1, chunks 2t or 2t + 1) read 8 different 16-byte units.  Scale
// boxes are swizzled (unit u of row r at u ^ (r mod 8)), so rows 0..7 read distinct banks.
// The activation is staged once per CTA (after the programmatic-launch wait; each warp
// stages only the blocks it uses, so no CTA-wide barrier) in MMA order: block kb, step q,
// chunk c at byte (kb * 32 + q * 8 + c) * 16, the 8 halves paired as the conversion pairs
// nibbles.
//
// Launch overlap.  When a CTA's whole share of the weights fits in half an SM's shared
// memory, the kernel runs 8 consumer warps with at most half the registers, so the next
// call's CTA can be resident on the same SM: its producer streams all of its stages before
// the programmatic-launch wait, while this call computes.  Larger problems run one CTA per
// SM with 16 consumer warps and a deeper ring.
//
// Every wait is bounded; a wait that gives up records its cause in the device status word
// and the affected tile's outputs are NaN.  Each tile's sum over warps is taken in warp
// order after a consumer barrier, so results are deterministic.
#include <cuda.h>
#include <cstring>
#include <cudaTypedefs.h>

#include "mma_sync.cuh"
#include "mnb_device.cuh"
#include "mnb_internal.h"
#include "tcgen05.cuh"

namespace mnb {
namespace {

constexpr int kRows = 16;     // weight rows per tile (the MMA's M)
constexpr int kBlockK = 256;  // k per block (8 chunks of 32)
constexpr int kRowPad = 16;   // staged packed row stride = slice bytes + 16
constexpr int kMaxStages = 8;
constexpr int kBoxBytes = 2048;  // one scale box: 16 rows x 128 bytes

struct MmaGemvArgs {
  const __half* A;
  const uint8_t* packed[2];
  const uint8_t* zp[2];
  void* Y;
  int K, N;
  int gshift;        // log2(bs / 32)
  int row_bytes;     // K / 2
  int kslice, nslices;
  int prow;          // kslice / 2 + kRowPad
  int sslice;        // scale bytes per row of a (full) slice
  int zrow;          // zero-point bytes per row (0: none); whole-K stages only
  int poff, zoff;    // packed rows and zero points inside a weight's sub-stage
  int wbytes;        // one weight's sub-stage (multiple of 1024)
  int stage_bytes;   // NWT * wbytes
  int stages;
  int ntiles;
  int ssz;           // bytes per scale
  uint32_t* status;
  const __half* bias;
  int bias_mode;
};

__device__ __forceinline__ float silu_f32(float x) { return x / (1.0f + expf(-x)); }

// 16-byte shared load into v when pred is set; v keeps its old contents otherwise.
__device__ __forceinline__ void lds128_pred(uint32_t (&v)[4], uint32_t addr, uint32_t pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "@p ld.shared.v4.u32 {%0,%1,%2,%3}, [%5];\n\t}"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3])
      : "r"(pred), "r"(addr)
      : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int q) {
  return q == 0 ? v.x : (q == 1 ? v.y : (q == 2 ? v.z : v.w));
}

// Shared address of byte o of row r in a weight sub-stage's swizzled scale boxes.
__device__ __forceinline__ uint32_t scale_addr(uint32_t wbase, int r, int o) {
  return wbase + (uint32_t)((o >> 7) * kBoxBytes + r * 128 + ((((o & 127) >> 4) ^ (r & 7)) << 4) + (o & 15));
}

// The two scales (chunks 2t and 2t + 1 of a block) of row r, as fp32.
template <bool S16, int CPG>
__device__ __forceinline__ void load_scales(uint32_t wbase, int r, int o0, float& s0, float& s1) {
  if constexpr (CPG == 1) {
    if constexpr (S16) {
      const uint32_t h = lds_u32_a(scale_addr(wbase, r, o0));
      s0 = half_bits_to_float(h & 0xffffu);
      s1 = half_bits_to_float(h >> 16);
    } else {
      const uint2 f = lds_u64_a(scale_addr(wbase, r, o0));
      s0 = __uint_as_float(f.x);
      s1 = __uint_as_float(f.y);
    }
  } else {
    s0 = S16 ? half_bits_to_float(lds_u16_a(scale_addr(wbase, r, o0))) : __uint_as_float(lds_u32_a(scale_addr(wbase, r, o0)));
    s1 = s0;
  }
}

template <int NCW, bool PAIR, bool S16, bool ZP, int CPG>
__global__ void __launch_bounds__((NCW + 1) * 32, (NCW <= 8 ? 2 : 1))
    gemv_mma_kernel(const MmaGemvArgs p, const __grid_constant__ CUtensorMap tmap0,
                    const __grid_constant__ CUtensorMap tmap1) {
  constexpr int NWT = PAIR ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ float red[2][NWT][NCW][kRows];
  __shared__ int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned (swizzled boxes)
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t act_u32 = ring_u32 + (uint32_t)(p.stages * p.stage_bytes);
  const int t_begin = (int)(((long long)blockIdx.x * p.ntiles) / gridDim.x);
  const int t_end = (int)(((long long)(blockIdx.x + 1) * p.ntiles) / gridDim.x);
  const int nst = (t_end - t_begin) * p.nslices;
  const int S = p.stages;
  const int bps = p.kslice / kBlockK;  // blocks in a full slice

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
    int slot = 0, issued = 0;
    uint32_t phase = 0;
    for (int st = 0; st < nst; ++st) {
      int free_slot = 1;
      if (lane == 0 && st >= S && !mbar_wait_bounded(&empty_bar[slot], phase ^ 1u)) {
        report_status(p.status, kStatusEmptyWait);
        atomicExch(&failed, 1);
        free_slot = 0;
      }
      if (!__shfl_sync(kFull, free_slot, 0)) break;
      const int ti = t_begin + st / p.nslices, si = st % p.nslices;
      const int n0 = ti * kRows, nr = min(kRows, p.N - n0);
      const int k0 = si * p.kslice, klen = min(p.kslice, p.K - k0);
      const int pbytes = klen >> 1;
      const int sb_slice = (klen >> (5 + p.gshift)) * p.ssz;  // scale bytes of this slice
      const int nsb = (sb_slice + 127) >> 7;
      const uint32_t bytes = (uint32_t)NWT * ((uint32_t)(nr * pbytes) + (uint32_t)(nsb * kBoxBytes) +
                                              (uint32_t)(ZP ? nr * p.zrow : 0));
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[slot], bytes);
      __syncwarp();
      uint8_t* stg = ring + (size_t)slot * p.stage_bytes;
#pragma unroll
      for (int wt = 0; wt < NWT; ++wt) {
        uint8_t* wb = stg + wt * p.wbytes;
        if (lane < nr)
          bulk_g2s(wb + p.poff + lane * p.prow, p.packed[wt] + (long long)(n0 + lane) * p.row_bytes + (k0 >> 1),
                   (uint32_t)pbytes, &full_bar[slot]);
        const CUtensorMap* tm = wt == 0 ? &tmap0 : &tmap1;
        for (int b = lane - 16; b >= 0 && b < nsb; b += 16)
          tc::tma_load_2d(wb + b * kBoxBytes, tm, si * p.sslice + b * 128, n0, &full_bar[slot]);
        if (ZP && lane == 0)
          bulk_g2s(wb + p.zoff, p.zp[wt] + (long long)n0 * p.zrow, (uint32_t)(nr * p.zrow), &full_bar[slot]);
      }
      issued = st + 1;
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    // Every copy issued must land before the CTA exits; after a failed wait this bounds it.
    if (lane == 0)
      for (int st = issued > S ? issued - S : 0; st < issued; ++st)
        (void)mbar_wait_bounded(&full_bar[st % S], (uint32_t)(st / S) & 1u);
    pdl_launch_dependents();
  } else {
    // ------------------------------- consumers ------------------------------------
    pdl_launch_dependents();
    const int g = lane >> 2, t = lane & 3;
    const uint32_t bdata = (uint32_t)((g >> 1) == t);  // this lane carries B column g
    pdl_wait();
    // Stage this warp's activation blocks in MMA order (lane l holds halves 8l .. 8l + 7 of
    // a block: chunk l / 4, step l % 4).
    for (int si = 0; si < p.nslices; ++si) {
      const int nb = (min(p.kslice, p.K - si * p.kslice)) / kBlockK;
      const int b_lo = (warp * nb) / NCW, b_hi = ((warp + 1) * nb) / NCW;
      for (int b0 = b_lo; b0 < b_hi; b0 += 4) {
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          x[u] = make_uint4(0, 0, 0, 0);
          const int kb = si * bps + b0 + u;
          if (b0 + u < b_hi) x[u] = *reinterpret_cast<const uint4*>(p.A + (long long)kb * kBlockK + 8 * lane);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (b0 + u < b_hi) {
            const int kb = si * bps + b0 + u;
            uint32_t q[4];
            pair_halves_stride4(x[u], q);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                             act_u32 + (uint32_t)((kb * 32 + (lane & 3) * 8 + (lane >> 2)) * 16)),
                         "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                         : "memory");
          }
        }
      }
    }
    __syncwarp();

    const uint32_t zl8 = zp_lo_const(8u), zh8 = zp_hi_const(8u);
    uint32_t bq[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) bq[q][0] = bq[q][1] = bq[q][2] = bq[q][3] = 0u;
    float acc[NWT][2];
    bool ok = true;
    int slot = 0;
    uint32_t phase = 0;
    for (int st = 0; st < nst; ++st) {
      const int tl = st / p.nslices, si = st % p.nslices;
      if (si == 0) {
#pragma unroll
        for (int wt = 0; wt < NWT; ++wt) acc[wt][0] = acc[wt][1] = 0.0f;
      }
      if (ok && !mbar_wait_bounded(&full_bar[slot], phase)) {
        report_status(p.status, kStatusFullWait);
        atomicExch(&failed, 1);
        ok = false;
      }
      const uint32_t sb = ring_u32 + (uint32_t)(slot * p.stage_bytes);
      const int nb = (min(p.kslice, p.K - si * p.kslice)) / kBlockK;
      const int b_lo = (warp * nb) / NCW, b_hi = ok ? ((warp + 1) * nb) / NCW : b_lo;
      for (int b = b_lo; b < b_hi; ++b) {
        const int kb = si * bps + b;
        const uint32_t abase = act_u32 + (uint32_t)(kb * 512 + g * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) lds128_pred(bq[q], abase + (uint32_t)(q * 128), bdata);
        // groups (within the slice) of chunks 2t and 2t + 1, and the scale byte offset
        const int c0 = 8 * b + 2 * t;
        const int gs0 = c0 >> p.gshift;
        const int o0 = gs0 * p.ssz;
#pragma unroll
        for (int wt = 0; wt < NWT; ++wt) {
          const uint32_t wbase = sb + (uint32_t)(wt * p.wbytes);
          const uint32_t ra = wbase + (uint32_t)(p.poff + g * p.prow + b * 128 + 32 * t);
          const uint32_t rb = ra + (uint32_t)(8 * p.prow);
          const uint4 xa = lds128_a(ra), ya = lds128_a(ra + 16u);
          const uint4 xb = lds128_a(rb), yb = lds128_a(rb + 16u);
          uint32_t zlxa = zl8, zhxa = zh8, zlya = zl8, zhya = zh8;
          uint32_t zlxb = zl8, zhxb = zh8, zlyb = zl8, zhyb = zh8;
          if constexpr (ZP) {
            const int gs1 = (c0 + 1) >> p.gshift;
            const uint32_t za = lds_u8_a(wbase + (uint32_t)(p.zoff + g * p.zrow + (gs0 >> 1)));
            const uint32_t zb = lds_u8_a(wbase + (uint32_t)(p.zoff + (g + 8) * p.zrow + (gs0 >> 1)));
            const uint32_t sh0 = (uint32_t)(gs0 & 1) * 4u, sh1 = (uint32_t)(gs1 & 1) * 4u;
            const uint32_t za0 = (za >> sh0) & 15u, za1 = (za >> sh1) & 15u;
            const uint32_t zb0 = (zb >> sh0) & 15u, zb1 = (zb >> sh1) & 15u;
            zlxa = zp_lo_const(za0);
            zhxa = zp_hi_const(za0);
            zlya = zp_lo_const(za1);
            zhya = zp_hi_const(za1);
            zlxb = zp_lo_const(zb0);
            zhxb = zp_hi_const(zb0);
            zlyb = zp_lo_const(zb1);
            zhyb = zp_hi_const(zb1);
          }
          float dx0[4], dx1[4], dy0[4], dy1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t da[4], db[4], ea[4], eb[4];
            nibbles_to_centered_half2(word_of(xa, q), zlxa, zhxa, da);
            nibbles_to_centered_half2(word_of(xb, q), zlxb, zhxb, db);
            nibbles_to_centered_half2(word_of(ya, q), zlya, zhya, ea);
            nibbles_to_centered_half2(word_of(yb, q), zlyb, zhyb, eb);
            if (q == 0) {
              mma16816_zero(dx0, da[0], db[0], da[1], db[1], bq[q][0], bq[q][1]);
              mma16816_zero(dx1, da[2], db[2], da[3], db[3], bq[q][2], bq[q][3]);
              mma16816_zero(dy0, ea[0], eb[0], ea[1], eb[1], bq[q][0], bq[q][1]);
              mma16816_zero(dy1, ea[2], eb[2], ea[3], eb[3], bq[q][2], bq[q][3]);
            } else {
              mma16816(dx0, da[0], db[0], da[1], db[1], bq[q][0], bq[q][1]);
              mma16816(dx1, da[2], db[2], da[3], db[3], bq[q][2], bq[q][3]);
              mma16816(dy0, ea[0], eb[0], ea[1], eb[1], bq[q][0], bq[q][1]);
              mma16816(dy1, ea[2], eb[2], ea[3], eb[3], bq[q][2], bq[q][3]);
            }
          }
          float sa0, sa1, sb0, sb1;
          load_scales<S16, CPG>(wbase, g, o0, sa0, sa1);
          load_scales<S16, CPG>(wbase, g + 8, o0, sb0, sb1);
          // lane (g, t): X column 2t (registers 0, 2) and Y column 2t + 1 (registers 1, 3)
          acc[wt][0] = fmaf(dx0[0] + dx1[0], sa0, acc[wt][0]);
          acc[wt][0] = fmaf(dy0[1] + dy1[1], sa1, acc[wt][0]);
          acc[wt][1] = fmaf(dx0[2] + dx1[2], sb0, acc[wt][1]);
          acc[wt][1] = fmaf(dy0[3] + dy1[3], sb1, acc[wt][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp no longer reads the slot
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
      if (si == p.nslices - 1) {
        // The tile is done: sum the four lanes of each row, then across warps in order.
        const int buf = tl & 1;
#pragma unroll
        for (int wt = 0; wt < NWT; ++wt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float v = acc[wt][h];
            v += __shfl_xor_sync(kFull, v, 1);
            v += __shfl_xor_sync(kFull, v, 2);
            if (t == 0) red[buf][wt][warp][g + 8 * h] = v;
          }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
        if (warp == tl % NCW && lane < kRows) {
          const int n = (t_begin + tl) * kRows + lane;
          if (n < p.N) {
            float v[NWT];
#pragma unroll
            for (int wt = 0; wt < NWT; ++wt) {
              float s = 0.0f;
#pragma unroll
              for (int w = 0; w < NCW; ++w) s += red[buf][wt][w][lane];
              v[wt] = s;
            }
            __half out;
            if constexpr (PAIR) out = __float2half_rn(silu_f32(v[0]) * v[1]);
            else out = round_out(v[0], p.bias, n, p.bias_mode);
            if (failed) out = __ushort_as_half(0x7e00);
            reinterpret_cast<__half*>(p.Y)[n] = out;
          }
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
using MmaKernel = void (*)(const MmaGemvArgs, const CUtensorMap, const CUtensorMap);

template <int NCW, bool PAIR, bool S16, bool ZP>
MmaKernel pick_cpg(int cpg) {
  if (cpg == 1) return gemv_mma_kernel<NCW, PAIR, S16, ZP, 1>;
  if (cpg == 2) return gemv_mma_kernel<NCW, PAIR, S16, ZP, 2>;
  if (cpg == 4) return gemv_mma_kernel<NCW, PAIR, S16, ZP, 4>;
  return nullptr;
}

template <int NCW, bool PAIR>
MmaKernel pick(bool s16, bool zp, int cpg) {
  if (s16) return zp ? pick_cpg<NCW, PAIR, true, true>(cpg) : pick_cpg<NCW, PAIR, true, false>(cpg);
  return zp ? pick_cpg<NCW, PAIR, false, true>(cpg) : pick_cpg<NCW, PAIR, false, false>(cpg);
}

// Dynamic shared memory per CTA when two CTAs share an SM (the calls overlap), and when one
// CTA has the SM.
constexpr int kHalfSmBudget = 100 * 1024;
constexpr int kFullSmBudget = 200 * 1024;

template <bool PAIR>
cudaError_t launch_mma_impl(LaunchCtx& ctx, const void* A, const QWeight* w, int K, int N, int bs, void* Y) {
  constexpr int NWT = PAIR ? 2 : 1;
  if (K % kBlockK != 0 || (bs != 32 && bs != 64 && bs != 128) || K % bs != 0) return cudaErrorNotSupported;
  if (PAIR && (w[0].scales_f16 != w[1].scales_f16 || (w[0].zp == nullptr) != (w[1].zp == nullptr)))
    return cudaErrorNotSupported;
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (encode == nullptr) return cudaErrorNotSupported;
  const bool s16 = w[0].scales_f16 != 0;
  const bool zp = w[0].zp != nullptr;
  const int ssz = s16 ? 2 : 4;
  const int G = K / bs;
  const int srow = G * ssz;
  if (srow % 16 != 0) return cudaErrorNotSupported;  // tensor-map row stride
  MmaGemvArgs a = {};
  a.A = static_cast<const __half*>(A);
  a.Y = Y;
  a.K = K;
  a.N = N;
  a.gshift = bs == 32 ? 0 : (bs == 64 ? 1 : 2);
  a.row_bytes = K / 2;
  a.ssz = ssz;
  a.zrow = zp ? (G + 1) / 2 : 0;
  a.ntiles = (N + kRows - 1) / kRows;
  // A partial last tile copies nr * zrow zero-point bytes: a 16-byte multiple is required.
  if (zp && ((N % kRows) * a.zrow) % 16 != 0) return cudaErrorNotSupported;
  for (int t = 0; t < 2; ++t) {
    const QWeight& q = w[t < NWT ? t : 0];
    a.packed[t] = q.packed;
    a.zp[t] = q.zp;
  }
  const int act_bytes = K * 2;
  // Sub-stage layout for a K slice of ks: [scale boxes][packed rows][zero points], 1024-aligned.
  auto layout = [&](int ks) {
    a.kslice = ks;
    a.nslices = (K + ks - 1) / ks;
    a.prow = ks / 2 + kRowPad;
    a.sslice = (ks / bs) * ssz;
    const int nsb = (a.sslice + 127) / 128;
    a.poff = nsb * kBoxBytes;
    a.zoff = a.poff + kRows * a.prow;
    a.wbytes = (a.zoff + kRows * a.zrow + 1023) / 1024 * 1024;
    a.stage_bytes = NWT * a.wbytes;
  };
  int grid = ctx.num_sms < a.ntiles ? ctx.num_sms : a.ntiles;
  const int max_tiles = (a.ntiles + grid - 1) / grid;
  // Two CTAs per SM when every stage of a CTA fits half the SM: all of its weights are then
  // requested at once, before the programmatic-launch wait.
  layout(K);
  bool half_sm = (size_t)max_tiles * a.stage_bytes + act_bytes + 1024 <= (size_t)kHalfSmBudget;
  if (half_sm) {
    a.stages = max_tiles;
  } else {
    // One CTA per SM: the whole K range per stage when two stages fit, else K slices (whole
    // 256-k blocks, scale bytes in whole boxes; no zero points).
    int ks = K;
    auto fits = [&]() { return 2 * (size_t)a.stage_bytes + act_bytes + 1024 <= (size_t)kFullSmBudget; };
    if (!fits()) {
      ks = 0;
      if (zp) return cudaErrorNotSupported;
      for (int cand = (K / 2) / kBlockK * kBlockK; cand >= 1024; cand -= kBlockK) {
        if (cand % bs != 0 || ((cand / bs) * ssz) % 128 != 0) continue;
        layout(cand);
        if (fits()) {
          ks = cand;
          break;
        }
      }
      if (ks == 0) return cudaErrorNotSupported;
    }
    a.stages = (int)((kFullSmBudget - act_bytes - 1024) / a.stage_bytes);
    if (a.stages > kMaxStages) a.stages = kMaxStages;
  }
  a.status = ctx.status;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = PAIR ? 0 : ctx.bias_mode;

  CUtensorMap tm[2];
  for (int t = 0; t < 2; ++t) {
    memset(&tm[t], 0, sizeof(CUtensorMap));
    const QWeight& q = w[t < NWT ? t : 0];
    const cuuint64_t gdim[2] = {(cuuint64_t)srow, (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)srow};
    const cuuint32_t box[2] = {128, (cuuint32_t)kRows};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm[t], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(q.scales), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
  }
  const int cpg = bs / 32;
  MmaKernel kern = half_sm ? pick<8, PAIR>(s16, zp, cpg) : pick<16, PAIR>(s16, zp, cpg);
  if (kern == nullptr) return cudaErrorNotSupported;
  const size_t smem = (size_t)a.stages * a.stage_bytes + act_bytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int threads = ((half_sm ? 8 : 16) + 1) * 32;
  ctx.variant = PAIR ? "gemv_pair_swiglu_mma" : "gemv_mma";
  return launch_kernel(ctx, kern, dim3(grid), dim3(threads), smem, a, tm[0], tm[1]);
}

}  // namespace

cudaError_t launch_gemv_mma(LaunchCtx& ctx, const void* A, const QWeight& w, int K, int N, int bs, void* Y) {
  return launch_mma_impl<false>(ctx, A, &w, K, N, bs, Y);
}

cudaError_t launch_gemv_pair_swiglu_mma(LaunchCtx& ctx, const void* A, const QWeight& gate, const QWeight& up,
                                        int K, int N, int bs, void* out) {
  const QWeight w[2] = {gate, up};
  return launch_mma_impl<true>(ctx, A, w, K, N, bs, out);
}

}  // namespace mnb
