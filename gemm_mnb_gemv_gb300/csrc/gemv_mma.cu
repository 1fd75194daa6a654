// M = 1 GEMV (and the paired gate/up SwiGLU GEMV) with the multiply-accumulate on the
// tensor cores: mma.sync m16n8k16, fp16 operands, fp32 accumulate.
//
// Why: a decode GEMV moves ~0.58 bytes per weight, and a CUDA-core inner loop (nibble
// conversion plus one mixed-precision FMA per weight) runs out of instruction issue before
// it runs out of bandwidth.  Here the conversion is the only per-weight CUDA-core work;
// the products and sums go to the tensor cores.
//
// Data flow.  A CTA owns a contiguous range of 16-row weight tiles (rows are output
// columns n).  A producer lane streams each tile into a ring of shared-memory stages, one
// weight and one K slice per stage, with three copies: the packed bytes as one 3-D tensor
// box (128 bytes x 16 rows x the slice's 128-byte segments), the scales as one 3-D box (or
// one 2-D box per 128 bytes when scale rows are not whole 128 bytes), the zero points of
// the tile's rows as one bulk copy.  Both boxes are 128-byte swizzled: 16-byte unit u of
// row r sits at unit u ^ (r mod 8) of its 128-byte line.  Consumer warps split each
// slice into blocks of 256 k (one packed segment, 8 chunks of 32 k).
//
// The MMA mapping.  Lane (g, t) (g = lane / 4, t = lane % 4) reads chunks 2t and 2t + 1 of
// a block from rows g and g + 8 and converts each 32-bit word into exact fp16 (code - zp)
// (magic-number conversion, zero point folded into its constants).  Word q of chunk 2t
// feeds the "X" MMAs of step q and word q of chunk 2t + 1 the "Y" MMAs, as the A operand
// (rows g, g + 8; the k order inside an MMA is the conversion's pairing, used identically
// for both operands).  The B operand holds the activation: column c of B carries chunk c
// of the block at the k slots of lane c / 2 and zero elsewhere, so in the X MMAs column 2t
// of D is row n's partial dot with chunk 2t, and in the Y MMAs column 2t + 1 is its partial
// dot with chunk 2t + 1; the other columns are never read.  Lane (g, t) therefore receives
// exactly the partial dots of its own chunks (D registers 0 and 2 of X, 1 and 3 of Y) and
// multiplies each by the scale of its group (scale after the partial dot of each
// 32-element chunk, as the fp16 GEMV of matmul_nbits.rs applies its per-block scale),
// accumulating in fp32.  Only 8 lanes of a warp load B; the other lanes keep zeros.
//
// Bank conflicts.  In a swizzled segment the 8 lanes of a quarter-warp (rows g, g + 1,
// chunk 2t or 2t + 1) read 8 different 16-byte units; rows g and g + 8 share a swizzle.
// The activation (K <= 8192) is staged once per CTA after the programmatic-launch wait, each
// warp only the blocks it uses (no CTA-wide barrier), in MMA order with the 8 halves of a
// step paired as the conversion pairs nibbles.  A larger one is not staged, so the weight
// stages keep the shared memory: each warp requests the lines of its blocks into L1, and
// the 8 lanes that carry B load their chunk (64 contiguous bytes per block) and pair it.
//
// Tile sums.  With one weight and at most S + 1 tiles per CTA (S ring stages), each lane
// posts its two row partials of a tile to the tile's own slot and, after a barrier of the
// consumer warps at the end, one warp per tile adds them in warp and lane order and stores
// it; otherwise each warp sums its four lanes per row first and the last warp to post a
// tile (a shared-memory counter) adds and stores it, so no warp waits on the others.
//
// Row mapping (speculative verify, 2 <= M <= 8 / G, G = 4 / CPG quant groups per four
// chunks: block sizes 32 and 64).  Lane (g, t) converts chunks t and t + 4 instead, so one
// MMA's k range spans four consecutive chunks; B column m * G + j carries activation row m
// on the k slots of group j and zeros elsewhere, and D column m * G + j is each weight
// row's partial dot with row m over group j: the same 16 MMAs per 4096 weights as M = 1.
//
// Launch overlap.  When a CTA's whole share fits half an SM (8 consumer warps, at most half
// the SM's registers and shared memory each), one CTA per SM per call: the next call's CTA
// is resident while this call runs and its producer streams all of its stages before the
// programmatic-launch wait.  Larger problems run two CTAs of the same call per SM when
// stages of at least 32 KB fit half an SM, else one CTA per SM with 16 consumer warps and
// a deeper ring.
//
// Every wait is bounded; a wait that gives up records its cause in the device status word
// and the affected tile's outputs are NaN.  Results are deterministic.
#include <cuda.h>
#include <cstring>
#include <cudaTypedefs.h>

#include "mma_sync.cuh"
#include "mnb_device.cuh"
#include "mnb_internal.h"
#include "tcgen05.cuh"

namespace mnb {
namespace {

constexpr int kRows = 16;        // weight rows per tile (the MMA's M)
constexpr int kBlockK = 256;     // k per block (8 chunks of 32): one 128-byte packed segment
constexpr int kMaxStages = 8;
constexpr int kBoxBytes = 2048;  // one swizzled box slab: 16 rows x 128 bytes
// tile-sum floats per warp and weight in a slot: 32 lanes x 2 rows (one weight, posted per
// lane), or the 16 rows (two weights, four lanes summed first)
template <bool PAIR>
constexpr int red_per_warp() { return PAIR ? kRows : 64; }

struct MmaGemvArgs {
  const __half* A;
  int M;             // activation rows (1: the GEMV mapping; 2 .. 2 * CPG: the row mapping)
  const uint8_t* zp[2];
  void* Y;
  int K, N;
  int kslice, nslices;
  int nseg;          // 128-byte packed segments (256 k) per row of a full slice
  int sslice;        // scale bytes per row of a full slice
  int s3d;           // scales copied as one 3-D box per stage (scale rows in whole 128 bytes)
  int nsbox;         // scale boxes (16 rows x 128 bytes) per stage
  int zrow;          // zero-point bytes per row (0: none); whole-K stages only
  int poff, zoff;    // packed segments and zero points inside a stage
  int stage_bytes;   // one stage: one weight's tile slice (multiple of 1024)
  int stages;
  int act_smem;      // 1: the activation is staged after the stages (K * 2 bytes), 0: read from L1/L2
  int red_off;       // tile-sum slots after the stages (and the activation): [stages + 1][weights][warps][64]
  int ntiles;
  uint32_t* status;
  const __half* bias;
  int bias_mode;
};

// One block's weight side for one lane: the packed words of chunks 2t (X) and 2t + 1 (Y) of
// rows g (a) and g + 8 (b), the conversion constants of their zero points and the scales.
struct BlockFrag {
  uint4 xa, ya, xb, yb;
  uint32_t zlxa, zhxa, zlya, zhya, zlxb, zhxb, zlyb, zhyb;
  float sa0, sa1, sb0, sb1;
};

// The row mapping's weight side of one block for one lane: the same 16 A-fragment words
// (chunks t and t + 4) and the scales of its two D columns' groups: X row g, Y row g, X row
// g + 8, Y row g + 8 (two each).
struct RowFrag {
  uint32_t w[4][16];
  float s[8];
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

// The two scales (chunks 2t and 2t + 1 of a block) at shared address `addr`, as fp32: for
// block size 32 two consecutive groups, otherwise one group.
template <bool S16, int CPG>
__device__ __forceinline__ void load_scales(uint32_t addr, float& s0, float& s1) {
  if constexpr (CPG == 1) {
    if constexpr (S16) {
      const uint32_t h = lds_u32_a(addr);
      s0 = half_bits_to_float(h & 0xffffu);
      s1 = half_bits_to_float(h >> 16);
    } else {
      const uint2 f = lds_u64_a(addr);
      s0 = __uint_as_float(f.x);
      s1 = __uint_as_float(f.y);
    }
  } else {
    s0 = S16 ? half_bits_to_float(lds_u16_a(addr)) : __uint_as_float(lds_u32_a(addr));
    s1 = s0;
  }
}

// CPG: 32-k chunks per quant group (1, 2, 4 for block sizes 32, 64, 128).  CPS: CTAs that
// share an SM (launch bounds leave each at most 1 / CPS of the registers).  ASM: the
// activation is staged in shared memory.  ROWS: 2 <= M <= 8 / G activation rows, G = 4 / CPG
// quant groups in four chunks (the row mapping below; block sizes 32 and 64).
template <int NCW, int CPS, bool PAIR, bool S16, bool ZP, int CPG, bool ASM, bool ROWS = false>
__global__ void __launch_bounds__((NCW + 1) * 32, CPS)
    gemv_mma_kernel(const MmaGemvArgs p, const __grid_constant__ CUtensorMap tmp0,
                    const __grid_constant__ CUtensorMap tmp1, const __grid_constant__ CUtensorMap tms0,
                    const __grid_constant__ CUtensorMap tms1) {
  constexpr int NWT = PAIR ? 2 : 1;
  constexpr int kSsz = S16 ? 2 : 4;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ unsigned red_cnt[kMaxStages + 1];
  __shared__ int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned (swizzled boxes)
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t act_u32 = ring_u32 + (uint32_t)(p.stages * p.stage_bytes);
  float* red = reinterpret_cast<float*>(ring + p.red_off);
  const int t_begin = (int)(((long long)blockIdx.x * p.ntiles) / gridDim.x);
  const int t_end = (int)(((long long)(blockIdx.x + 1) * p.ntiles) / gridDim.x);
  const int nsub = NWT * p.nslices;  // stages per tile: weight-major, then K slice
  const int nst = (t_end - t_begin) * nsub;
  const int S = p.stages;
  const int bps = p.kslice / kBlockK;  // blocks in a full slice

  if (tid == 0) {
    failed = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NCW);
    }
    for (int s = 0; s <= S; ++s) red_cnt[s] = 0u;
    fence_mbar_init();
  }
  __syncthreads();

  // Requests stage st (tile, weight, K slice) into ring slot `slot`.
  auto issue = [&](int st, int slot) {
    const int r = st % nsub;
    const int ti = t_begin + st / nsub, wt = r / p.nslices, si = r % p.nslices;
    const int n0 = ti * kRows, nr = min(kRows, p.N - n0);
    const int klen = min(p.kslice, p.K - si * p.kslice);
    const int nsb = p.s3d ? p.nsbox : (((klen / (32 * CPG)) * kSsz + 127) >> 7);
    const uint32_t bytes = (uint32_t)((p.nseg + nsb) * kBoxBytes) + (uint32_t)(ZP ? nr * p.zrow : 0);
    const bool w1 = NWT == 2 && wt == 1;
    uint8_t* wb = ring + (size_t)slot * p.stage_bytes;
    mbar_arrive_expect_tx(&full_bar[slot], bytes);
    // rows past N and segments past K arrive as zeros (and count in full)
    tc::tma_load_3d(wb + p.poff, w1 ? &tmp1 : &tmp0, 0, n0, si * bps, &full_bar[slot]);
    if (p.s3d)
      tc::tma_load_3d(wb, w1 ? &tms1 : &tms0, 0, n0, (si * p.sslice) >> 7, &full_bar[slot]);
    else
      for (int b = 0; b < nsb; ++b)
        tc::tma_load_2d(wb + b * kBoxBytes, w1 ? &tms1 : &tms0, si * p.sslice + b * 128, n0, &full_bar[slot]);
    if (ZP)
      bulk_g2s(wb + p.zoff, (w1 ? p.zp[1] : p.zp[0]) + (long long)n0 * p.zrow, (uint32_t)(nr * p.zrow),
               &full_bar[slot]);
  };
  // Adds the consumer warps' posted partials of tile tl (slot rp) in warp order (per lane:
  // lanes 4r', 4r' + 1, 4r' + 2, 4r' + 3 of row r = r' + 8h in turn) and stores the tile's
  // outputs (lanes 0..15).
  auto store_tile = [&](int tl, const float* rp, bool per_lane) {
    if constexpr (ROWS) {
      // output (m, r): lanes (r mod 8, t) of every warp whose columns 2t, 2t + 1 belong to row
      // m, in warp then lane order
      constexpr int G = 4 / CPG;
      for (int o = lane; o < kRows * p.M; o += 32) {
        const int r = o & (kRows - 1), m = o / kRows, n = (t_begin + tl) * kRows + r;
        if (n >= p.N) continue;
        float sum = 0.0f;
#pragma unroll
        for (int ww = 0; ww < NCW; ++ww)
#pragma unroll
          for (int tt = 0; tt < 4; ++tt)
            if ((2 * tt) / G == m) sum += *(volatile const float*)&rp[(ww * 32 + 4 * (r & 7) + tt) * 2 + (r >> 3)];
        __half out = round_out(sum, p.bias, n, p.bias_mode);
        if (*(volatile int*)&failed) out = __ushort_as_half(0x7e00);
        reinterpret_cast<__half*>(p.Y)[(long long)m * p.N + n] = out;
      }
      return;
    }
    const int n = (t_begin + tl) * kRows + lane;
    if (lane < kRows && n < p.N) {
      float v[NWT];
#pragma unroll
      for (int w = 0; w < NWT; ++w) {
        float sum = 0.0f;
        if (per_lane) {
          const int gg = lane & 7, hh = lane >> 3;
#pragma unroll
          for (int ww = 0; ww < NCW; ++ww)
#pragma unroll
            for (int tt = 0; tt < 4; ++tt)
              sum += *(volatile const float*)&rp[((w * NCW + ww) * 32 + 4 * gg + tt) * 2 + hh];
        } else {
#pragma unroll
          for (int ww = 0; ww < NCW; ++ww) sum += *(volatile const float*)&rp[(w * NCW + ww) * kRows + lane];
        }
        v[w] = sum;
      }
      __half out;
      if constexpr (PAIR) out = __float2half_rn(silu_f32(v[0]) * v[1]);
      else out = round_out(v[0], p.bias, n, p.bias_mode);
      if (*(volatile int*)&failed) out = __ushort_as_half(0x7e00);
      reinterpret_cast<__half*>(p.Y)[n] = out;
    }
  };
  if (warp == NCW) {
    // ------------------------------- producer -------------------------------------
    if (lane == 0) {
      int slot = 0, issued = 0;
      uint32_t phase = 0;
      for (int st = 0; st < nst; ++st) {
        if (st >= S && !mbar_wait_bounded(&empty_bar[slot], phase ^ 1u)) {
          report_status(p.status, kStatusEmptyWait);
          atomicExch(&failed, 1);
          break;
        }
        issue(st, slot);
        issued = st + 1;
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // Every copy issued must land before the CTA exits; after a failed wait this bounds it.
      for (int st = issued > S ? issued - S : 0; st < issued; ++st)
        (void)mbar_wait_bounded(&full_bar[st % S], (uint32_t)(st / S) & 1u);
    }
    __syncwarp();
    pdl_launch_dependents();
  } else {
    // ------------------------------- consumers ------------------------------------
    pdl_launch_dependents();
    const int g = lane >> 2, t = lane & 3;
    const uint32_t bdata = (uint32_t)((g >> 1) == t);  // this lane carries B column g
    // Per-lane group geometry of chunks 2t and 2t + 1 of block b (compile-time block size):
    // zero-point byte zb0 + zbs * b with the nibbles at shifts zsh0, zsh1; scale byte
    // so0 + sos * b within the slice's scale boxes.
    const int zb0 = CPG == 1 ? t : (CPG == 2 ? (t >> 1) : 0);
    const int zbs = CPG == 1 ? 4 : (CPG == 2 ? 2 : 1);
    const uint32_t zsh0 = CPG == 1 ? 0u : (CPG == 2 ? 4u * (uint32_t)(t & 1) : 4u * (uint32_t)((t >> 1) & 1));
    const uint32_t zsh1 = CPG == 1 ? 4u : zsh0;
    const int so0 = (CPG == 1 ? 2 * t : (CPG == 2 ? t : (t >> 1))) * kSsz;
    const int sos = (CPG == 1 ? 8 : (CPG == 2 ? 4 : 2)) * kSsz;
    const uint32_t zl8 = zp_lo_const(8u), zh8 = zp_hi_const(8u);
    // Block b of the stage at wbase, weight side: rows g and g + 8, chunks 2t (X) and 2t + 1
    // (Y), their zero points' conversion constants and their scales.
    auto prep = [&](uint32_t wbase, int b, BlockFrag& f) {
      const int o0 = so0 + sos * b;  // scale byte within the slice's boxes
      const uint32_t soff = (uint32_t)((o0 >> 7) * kBoxBytes + g * 128 + ((((o0 & 127) >> 4) ^ g) << 4) + (o0 & 15));
      // segment b, row g, 16-byte units 2t (X) and 2t + 1 (Y) swizzled by the row; row g + 8
      // 1024 bytes on, same swizzle
      const uint32_t seg = wbase + (uint32_t)(p.poff + b * kBoxBytes + g * 128);
      const uint32_t rxa = seg + (uint32_t)(((2 * t) ^ g) << 4), rya = seg + (uint32_t)(((2 * t + 1) ^ g) << 4);
      f.xa = lds128_a(rxa);
      f.ya = lds128_a(rya);
      f.xb = lds128_a(rxa + 1024u);
      f.yb = lds128_a(rya + 1024u);
      load_scales<S16, CPG>(wbase + soff, f.sa0, f.sa1);
      load_scales<S16, CPG>(wbase + soff + 1024u, f.sb0, f.sb1);  // row g + 8: same swizzle
      f.zlxa = f.zlya = f.zlxb = f.zlyb = zl8;
      f.zhxa = f.zhya = f.zhxb = f.zhyb = zh8;
      if constexpr (ZP) {
        const uint32_t zaddr = wbase + (uint32_t)(p.zoff + g * p.zrow + zb0 + zbs * b);
        const uint32_t za = lds_u8_a(zaddr), zb = lds_u8_a(zaddr + (uint32_t)(8 * p.zrow));
        const uint32_t za0 = (za >> zsh0) & 15u, za1 = (za >> zsh1) & 15u;
        const uint32_t zb0v = (zb >> zsh0) & 15u, zb1v = (zb >> zsh1) & 15u;
        f.zlxa = zp_lo_const(za0);
        f.zhxa = zp_hi_const(za0);
        f.zlya = zp_lo_const(za1);
        f.zhya = zp_hi_const(za1);
        f.zlxb = zp_lo_const(zb0v);
        f.zhxb = zp_hi_const(zb0v);
        f.zlyb = zp_lo_const(zb1v);
        f.zhyb = zp_hi_const(zb1v);
      }
    };
    // The activation side of 256-k block kb and the MMAs; adds the scaled partial dots of
    // rows g and g + 8 into vg and v8.  B column g holds chunk g of the block (halves 32g ..
    // 32g + 31; step q its 8 halves from 32g + 8q), paired as the conversion pairs nibbles,
    // on the lanes with g / 2 == t; the other lanes hold zeros.  Staged in shared memory, the
    // block sits in MMA order: step q, chunk c at byte (kb * 32 + q * 8 + c) * 16.
    auto finish = [&](int kb, const BlockFrag& f, float& vg, float& v8) {
      uint32_t bq[4][4];
      if constexpr (ASM) {
        const uint32_t abase = act_u32 + (uint32_t)(kb * 512 + g * 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          bq[q][0] = bq[q][1] = bq[q][2] = bq[q][3] = 0u;
          lds128_pred(bq[q], abase + (uint32_t)(q * 128), bdata);
        }
      } else {
        uint4 av[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) av[q] = make_uint4(0u, 0u, 0u, 0u);
        if (bdata) {
          const uint4* ap = reinterpret_cast<const uint4*>(p.A + (long long)kb * kBlockK + 32 * g);
#pragma unroll
          for (int q = 0; q < 4; ++q) av[q] = ap[q];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) pair_halves_stride4(av[q], bq[q]);
      }
      // step q: its four words converted to A fragments right before its four MMAs; one
      // accumulator for the X MMAs and one for the Y MMAs (eight MMAs each per block)
      float dx[4], dy[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t da[4], db[4], ea[4], eb[4];
        nibbles_to_centered_half2(word_of(f.xa, q), f.zlxa, f.zhxa, da);
        nibbles_to_centered_half2(word_of(f.xb, q), f.zlxb, f.zhxb, db);
        nibbles_to_centered_half2(word_of(f.ya, q), f.zlya, f.zhya, ea);
        nibbles_to_centered_half2(word_of(f.yb, q), f.zlyb, f.zhyb, eb);
        if (q == 0) {
          mma16816_zero(dx, da[0], db[0], da[1], db[1], bq[q][0], bq[q][1]);
          mma16816_zero(dy, ea[0], eb[0], ea[1], eb[1], bq[q][0], bq[q][1]);
        } else {
          mma16816(dx, da[0], db[0], da[1], db[1], bq[q][0], bq[q][1]);
          mma16816(dy, ea[0], eb[0], ea[1], eb[1], bq[q][0], bq[q][1]);
        }
        mma16816(dx, da[2], db[2], da[3], db[3], bq[q][2], bq[q][3]);
        mma16816(dy, ea[2], eb[2], ea[3], eb[3], bq[q][2], bq[q][3]);
      }
      // lane (g, t): X column 2t (registers 0, 2) and Y column 2t + 1 (registers 1, 3)
      vg = fmaf(dx[0], f.sa0, vg);
      vg = fmaf(dy[1], f.sa1, vg);
      v8 = fmaf(dx[2], f.sb0, v8);
      v8 = fmaf(dy[3], f.sb1, v8);
    };

    // Row mapping (ROWS): lane (g, t) converts chunks t (X) and t + 4 (Y) of rows g, g + 8, so
    // one MMA's k range spans four consecutive chunks, G = 4 / CPG quant groups; B column
    // m * G + j carries activation row m on the k slots of the chunks of group j (lanes t with
    // t / CPG == j) and zeros elsewhere, so column m * G + j of D is each row's partial dot
    // with row m over group j.  Lane (g, t) receives columns 2t, 2t + 1: activation row
    // (2t) / G, groups (2t) mod G and the next.
    constexpr int kG = 4 / CPG;
    const int mb = g / kG;  // activation row of B column g
    const uint32_t carrier = (uint32_t)(ROWS && g < p.M * kG && (t / CPG) == (g % kG));
    const uint32_t bsw = (uint32_t)((mb & 1) << 2);
    // zero-point bytes of chunks t, t + 4 of block b: rzx / rzy + rzs * b, nibble at rzsh
    const int rzx = CPG == 1 ? (t >> 1) : 0, rzy = CPG == 1 ? 2 + (t >> 1) : 1, rzs = CPG == 1 ? 4 : 2;
    const uint32_t rzsh = CPG == 1 ? 4u * (uint32_t)(t & 1) : 4u * (uint32_t)((t >> 1) & 1);
    // scale bytes of the lane's two X groups and two Y groups of block b
    const int rsx = (CPG == 1 ? 2 * (t & 1) : 0) * kSsz, rsy = rsx + (CPG == 1 ? 4 : 2) * kSsz;
    const int rss = (CPG == 1 ? 8 : 4) * kSsz;
    auto sw_off = [&](int o) -> uint32_t {  // swizzled offset of scale byte o (row g)
      return (uint32_t)((o >> 7) * kBoxBytes + g * 128 + ((((o & 127) >> 4) ^ g) << 4) + (o & 15));
    };
    auto prep_rows = [&](uint32_t wbase, int b, RowFrag& f) {
      const uint32_t seg = wbase + (uint32_t)(p.poff + b * kBoxBytes + g * 128);
      const uint32_t rxa = seg + (uint32_t)((t ^ g) << 4), rya = seg + (uint32_t)(((t + 4) ^ g) << 4);
      const uint4 xa = lds128_a(rxa), ya = lds128_a(rya);
      const uint4 xb = lds128_a(rxa + 1024u), yb = lds128_a(rya + 1024u);
      const uint32_t ox = sw_off(rsx + rss * b), oy = sw_off(rsy + rss * b);
      load_scales<S16, 1>(wbase + ox, f.s[0], f.s[1]);
      load_scales<S16, 1>(wbase + oy, f.s[2], f.s[3]);
      load_scales<S16, 1>(wbase + ox + 1024u, f.s[4], f.s[5]);  // row g + 8: same swizzle
      load_scales<S16, 1>(wbase + oy + 1024u, f.s[6], f.s[7]);
      uint32_t zlxa = zl8, zhxa = zh8, zlya = zl8, zhya = zh8;
      uint32_t zlxb = zl8, zhxb = zh8, zlyb = zl8, zhyb = zh8;
      if constexpr (ZP) {
        const uint32_t zrow = wbase + (uint32_t)(p.zoff + g * p.zrow + rzs * b);
        const uint32_t zxa = (lds_u8_a(zrow + (uint32_t)rzx) >> rzsh) & 15u;
        const uint32_t zya = (lds_u8_a(zrow + (uint32_t)rzy) >> rzsh) & 15u;
        const uint32_t zxb = (lds_u8_a(zrow + (uint32_t)(rzx + 8 * p.zrow)) >> rzsh) & 15u;
        const uint32_t zyb = (lds_u8_a(zrow + (uint32_t)(rzy + 8 * p.zrow)) >> rzsh) & 15u;
        zlxa = zp_lo_const(zxa);
        zhxa = zp_hi_const(zxa);
        zlya = zp_lo_const(zya);
        zhya = zp_hi_const(zya);
        zlxb = zp_lo_const(zxb);
        zhxb = zp_hi_const(zxb);
        zlyb = zp_lo_const(zyb);
        zhyb = zp_hi_const(zyb);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        nibbles_to_centered_half2(word_of(xa, q), zlxa, zhxa, f.w[q] + 0);
        nibbles_to_centered_half2(word_of(xb, q), zlxb, zhxb, f.w[q] + 4);
        nibbles_to_centered_half2(word_of(ya, q), zlya, zhya, f.w[q] + 8);
        nibbles_to_centered_half2(word_of(yb, q), zlyb, zhyb, f.w[q] + 12);
      }
    };
    // The staged activation of the row mapping: block kb, step q, row m, chunk c at 16-byte
    // entry ((kb * 4 + q) * M + m) * 8 + (c ^ 4 (m mod 2)), the halves paired as the
    // conversion pairs nibbles (the carriers of one step read distinct bank groups).
    auto finish_rows = [&](int kb, const RowFrag& f, float& vg, float& v8) {
      uint32_t bx[4][4], by[4][4];
      const uint32_t base = act_u32 + (uint32_t)((kb * 4 * p.M + mb) * 8 * 16);
      const uint32_t qs = (uint32_t)(p.M * 8 * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        bx[q][0] = bx[q][1] = bx[q][2] = bx[q][3] = 0u;
        by[q][0] = by[q][1] = by[q][2] = by[q][3] = 0u;
        lds128_pred(bx[q], base + q * qs + (((uint32_t)t ^ bsw) << 4), carrier);
        lds128_pred(by[q], base + q * qs + (((uint32_t)(t + 4) ^ bsw) << 4), carrier);
      }
      float x0[4], x1[4], y0[4], y1[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t* da = f.w[q];
        const uint32_t* db = f.w[q] + 4;
        const uint32_t* ea = f.w[q] + 8;
        const uint32_t* eb = f.w[q] + 12;
        if (q == 0) {
          mma16816_zero(x0, da[0], db[0], da[1], db[1], bx[q][0], bx[q][1]);
          mma16816_zero(x1, da[2], db[2], da[3], db[3], bx[q][2], bx[q][3]);
          mma16816_zero(y0, ea[0], eb[0], ea[1], eb[1], by[q][0], by[q][1]);
          mma16816_zero(y1, ea[2], eb[2], ea[3], eb[3], by[q][2], by[q][3]);
        } else {
          mma16816(x0, da[0], db[0], da[1], db[1], bx[q][0], bx[q][1]);
          mma16816(x1, da[2], db[2], da[3], db[3], bx[q][2], bx[q][3]);
          mma16816(y0, ea[0], eb[0], ea[1], eb[1], by[q][0], by[q][1]);
          mma16816(y1, ea[2], eb[2], ea[3], eb[3], by[q][2], by[q][3]);
        }
      }
      // registers 0, 1: row g, columns 2t, 2t + 1; registers 2, 3: row g + 8
      vg = fmaf(x0[0] + x1[0], f.s[0], vg);
      vg = fmaf(x0[1] + x1[1], f.s[1], vg);
      vg = fmaf(y0[0] + y1[0], f.s[2], vg);
      vg = fmaf(y0[1] + y1[1], f.s[3], vg);
      v8 = fmaf(x0[2] + x1[2], f.s[4], v8);
      v8 = fmaf(x0[3] + x1[3], f.s[5], v8);
      v8 = fmaf(y0[2] + y1[2], f.s[6], v8);
      v8 = fmaf(y0[3] + y1[3], f.s[7], v8);
    };

    pdl_wait();
    if constexpr (ROWS) {
      // Stage this warp's blocks of every activation row (lane l: halves 8l .. 8l + 7 of a
      // block, chunk l / 4, step l % 4), up to eight (block, row) loads in flight per lane.
      const int q = lane & 3, c = lane >> 2;
      for (int si = 0; si < p.nslices; ++si) {
        const int nb = (min(p.kslice, p.K - si * p.kslice)) / kBlockK;
        const int b_lo = (warp * nb) / NCW, b_hi = ((warp + 1) * nb) / NCW;
        // (block, row) pairs, row-minor, eight at a time: all loads, then all stores
        for (int b0 = b_lo, m0 = 0; b0 < b_hi;) {
          uint4 x[8];
          int bb = b0, mm = m0;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            x[u] = make_uint4(0, 0, 0, 0);
            if (bb < b_hi)
              x[u] = *reinterpret_cast<const uint4*>(p.A + (long long)mm * p.K + (long long)(si * bps + bb) * kBlockK + 8 * lane);
            if (++mm == p.M) {
              mm = 0;
              ++bb;
            }
          }
          bb = b0;
          mm = m0;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (bb < b_hi) {
              uint32_t w4[4];
              pair_halves_stride4(x[u], w4);
              const int e = (((si * bps + bb) * 4 + q) * p.M + mm) * 8 + (c ^ ((mm & 1) << 2));
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(act_u32 + (uint32_t)(e * 16)), "r"(w4[0]),
                           "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                           : "memory");
            }
            if (++mm == p.M) {
              mm = 0;
              ++bb;
            }
          }
          b0 = bb;
          m0 = mm;
        }
      }
      __syncwarp();
    } else if constexpr (ASM) {
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
    } else {
      // The activation is read from global memory by the lanes that carry B; this warp's lines
      // are first requested into L1 so that the first conversions overlap their latency.
      for (int si = 0; si < p.nslices; ++si) {
        const int nb = (min(p.kslice, p.K - si * p.kslice)) / kBlockK;
        const int b_lo = (warp * nb) / NCW, b_hi = ((warp + 1) * nb) / NCW;
        for (int i = lane; i < 4 * (b_hi - b_lo); i += 32)
          prefetch_l1(p.A + (long long)(si * bps + b_lo) * kBlockK + 64 * i);
      }
    }
    const int ntl = t_end - t_begin;
    bool ok = true;
    // Tile sums.  With at most S + 1 tiles every tile has its own slot, and the warps'
    // partials are added once after the last tile (no per-tile synchronisation).  Otherwise
    // slots are reused every S + 1 tiles and the last warp to post a tile adds and stores it;
    // the ring slot of a tile's last stage is released only after the post, so no warp can be
    // S + 1 tiles ahead of the warp that reads a slot.
    const bool deferred = ntl <= S + 1;
    const bool ring = nst > S;  // stages reuse ring slots: the producer waits for them to empty
    const bool per_lane = deferred && NWT == 1;
    int slot = 0;
    uint32_t phase = 0;
    for (int tl = 0; tl < ntl; ++tl) {
      float acc[NWT][2];
      int last_slot = 0;
#pragma unroll
      for (int wt = 0; wt < NWT; ++wt) {
        acc[wt][0] = acc[wt][1] = 0.0f;
        for (int si = 0; si < p.nslices; ++si) {
          // (a phase that completed long ago is seen by test_wait without the try_wait round trip)
          if (ok && !mbar_test_wait(&full_bar[slot], phase) && !mbar_wait_bounded(&full_bar[slot], phase)) {
            report_status(p.status, kStatusFullWait);
            atomicExch(&failed, 1);
            ok = false;
          }
          const uint32_t wbase = ring_u32 + (uint32_t)(slot * p.stage_bytes);
          const int nb = (min(p.kslice, p.K - si * p.kslice)) / kBlockK;
          const int b_lo = (warp * nb) / NCW, b_hi = ok ? ((warp + 1) * nb) / NCW : b_lo;
          float vg = 0.0f, v8 = 0.0f;  // this stage's partial sums of rows g and g + 8
          for (int b = b_lo; b < b_hi; ++b) {
            if constexpr (ROWS) {
              RowFrag f;
              prep_rows(wbase, b, f);
              finish_rows(si * bps + b, f, vg, v8);
            } else {
              BlockFrag f;
              prep(wbase, b, f);
              finish(si * bps + b, f, vg, v8);
            }
          }
          acc[wt][0] += vg;
          acc[wt][1] += v8;
          if (wt == NWT - 1 && si == p.nslices - 1) {
            last_slot = slot;
          } else if (ring) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp no longer reads the slot
          }
          if (++slot == S) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Post this warp's partials of the tile: per lane for one weight when every tile has its
      // own slot (they are added after the last tile), else the four lanes of each row summed
      // first.
      const int rs = deferred ? tl : tl % (S + 1);
      float* rp = red + (size_t)rs * (NWT * NCW * red_per_warp<PAIR>());
      if (per_lane) {
#pragma unroll
        for (int w = 0; w < NWT; ++w)
          *reinterpret_cast<float2*>(&rp[((w * NCW + warp) * 32 + lane) * 2]) = make_float2(acc[w][0], acc[w][1]);
      } else {
#pragma unroll
        for (int w = 0; w < NWT; ++w) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x = acc[w][h];
            x += __shfl_xor_sync(kFull, x, 1);
            x += __shfl_xor_sync(kFull, x, 2);
            if (t == 0) rp[(w * NCW + warp) * kRows + g + 8 * h] = x;
          }
        }
        __syncwarp();
        if (!deferred) {
          unsigned last = 0;
          if (lane == 0) {
            __threadfence_block();
            last = atomicInc(&red_cnt[rs], (unsigned)(NCW - 1)) == (unsigned)(NCW - 1);  // wraps to 0
          }
          last = __shfl_sync(kFull, last, 0);
          if (last) {
            __threadfence_block();
            store_tile(tl, rp, false);
          }
          __syncwarp();
        }
      }
      if (ring && lane == 0) mbar_arrive(&empty_bar[last_slot]);
    }
    if (deferred) {
      // every consumer warp has posted every tile: add and store them, one warp per tile
      asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
      for (int tl = warp; tl < ntl; tl += NCW) store_tile(tl, red + (size_t)tl * (NWT * NCW * red_per_warp<PAIR>()), per_lane);
    }
  }
}

// ----------------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------------
using MmaKernel = void (*)(const MmaGemvArgs, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                           const CUtensorMap);

// Consumer warps: 8 when two CTAs share an SM, else 16.
constexpr int kNcwTwo = 8, kNcwOne = 16;

template <int CPS, bool PAIR, bool S16, bool ZP, bool ASM>
MmaKernel pick_cpg(int cpg) {
  constexpr int NCW = CPS > 1 ? kNcwTwo : kNcwOne;
  if (cpg == 1) return gemv_mma_kernel<NCW, CPS, PAIR, S16, ZP, 1, ASM>;
  if (cpg == 2) return gemv_mma_kernel<NCW, CPS, PAIR, S16, ZP, 2, ASM>;
  if (cpg == 4) return gemv_mma_kernel<NCW, CPS, PAIR, S16, ZP, 4, ASM>;
  return nullptr;
}

// The row mapping: two CTAs per SM, staged activations, block sizes 32 and 64.
MmaKernel pick_rows(bool s16, bool zp, int cpg) {
  constexpr int N8 = kNcwTwo;
  if (cpg == 1) {
    if (s16) return zp ? gemv_mma_kernel<N8, 2, false, true, true, 1, true, true> : gemv_mma_kernel<N8, 2, false, true, false, 1, true, true>;
    return zp ? gemv_mma_kernel<N8, 2, false, false, true, 1, true, true> : gemv_mma_kernel<N8, 2, false, false, false, 1, true, true>;
  }
  if (cpg == 2) {
    if (s16) return zp ? gemv_mma_kernel<N8, 2, false, true, true, 2, true, true> : gemv_mma_kernel<N8, 2, false, true, false, 2, true, true>;
    return zp ? gemv_mma_kernel<N8, 2, false, false, true, 2, true, true> : gemv_mma_kernel<N8, 2, false, false, false, 2, true, true>;
  }
  return nullptr;
}

template <int CPS, bool PAIR, bool ASM>
MmaKernel pick(bool s16, bool zp, int cpg) {
  if (s16) return zp ? pick_cpg<CPS, PAIR, true, true, ASM>(cpg) : pick_cpg<CPS, PAIR, true, false, ASM>(cpg);
  return zp ? pick_cpg<CPS, PAIR, false, true, ASM>(cpg) : pick_cpg<CPS, PAIR, false, false, ASM>(cpg);
}

// Dynamic shared memory per CTA when two CTAs share an SM, and when one CTA has the SM; the
// stage size aimed at (several stages in flight per CTA).
constexpr int kTwoBudget = 100 * 1024;
constexpr int kOneBudget = 200 * 1024;
constexpr int kStageTargetTwo = 40 * 1024;
constexpr int kStageTargetOne = 72 * 1024;
constexpr int kTwoMinStage = 32 * 1024;
constexpr int kActSmemMax = 16 * 1024;  // activations staged in shared memory up to K = 8192
constexpr int kTwoBudgetRows = 110 * 1024;   // the row mapping (its activation rows are larger)
constexpr int kActSmemMaxRows = 32 * 1024;

// ROWS: 2 <= M <= 8 / G activation rows in the row mapping (M = 1 otherwise).
template <bool PAIR, bool ROWS = false>
cudaError_t launch_mma_impl(LaunchCtx& ctx, const void* A, const QWeight* w, int K, int N, int bs, void* Y,
                            int M = 1) {
  constexpr int NWT = PAIR ? 2 : 1;
  if (K % kBlockK != 0 || (bs != 32 && bs != 64 && bs != 128) || K % bs != 0) return cudaErrorNotSupported;
  if (ROWS && (PAIR || bs > 64 || M < 2 || M > 2 * (bs / 32) || (long long)M * K * 2 > kActSmemMaxRows))
    return cudaErrorNotSupported;
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
  a.M = ROWS ? M : 1;
  a.Y = Y;
  a.K = K;
  a.N = N;
  a.zrow = zp ? (G + 1) / 2 : 0;
  a.ntiles = (N + kRows - 1) / kRows;
  // A partial last tile copies nr * zrow zero-point bytes: a 16-byte multiple is required.
  if (zp && ((N % kRows) * a.zrow) % 16 != 0) return cudaErrorNotSupported;
  for (int t = 0; t < 2; ++t) a.zp[t] = w[t < NWT ? t : 0].zp;
  // Stage layout for a K slice of ks: [scale boxes][packed segments][zero points], 1024-aligned.
  auto layout = [&](int ks) {
    a.kslice = ks;
    a.nslices = (K + ks - 1) / ks;
    a.nseg = ks / kBlockK;
    a.sslice = (ks / bs) * ssz;
    a.nsbox = (a.sslice + 127) / 128;
    a.poff = a.nsbox * kBoxBytes;
    a.zoff = a.poff + a.nseg * kBoxBytes;
    a.stage_bytes = (a.zoff + kRows * a.zrow + 1023) / 1024 * 1024;
  };
  // The K slice: the whole K range when its stage is at most `target`, else the largest
  // slice (whole 256-k blocks and quant groups, scale bytes in whole 128 bytes; not with
  // zero points) that is, else the smallest such slice.  False if there is none.
  auto choose = [&](int target) {
    layout(K);
    if (a.stage_bytes <= target || zp) return true;  // zero points: whole-K stages only
    int smallest = 0;
    for (int cand = (K - 1) / kBlockK * kBlockK; cand >= kBlockK; cand -= kBlockK) {
      if (cand % bs != 0 || ((cand / bs) * ssz) % 128 != 0) continue;
      smallest = cand;
      layout(cand);
      if (a.stage_bytes <= target) return true;
    }
    if (smallest == 0) return false;
    layout(smallest);
    return true;
  };
  // Launch shape, in order of preference:
  //  * two CTAs per SM, one CTA per SM per call, when all of a CTA's stages fit half an SM;
  //  * two CTAs of the same call per SM when stages of at least kTwoMinStage fit half an SM
  //    (two stages in flight per CTA, sixteen warps computing per SM);
  //  * else one CTA per SM with sixteen consumer warps and a deeper ring.
  // each stage also needs one tile-sum slot (plus one spare slot)
  const int rps_two = NWT * kNcwTwo * red_per_warp<PAIR>() * 4, rps_one = NWT * kNcwOne * red_per_warp<PAIR>() * 4;
  int grid = 0, cps = 0;
  // The activation is staged in shared memory when it is small; larger ones are read
  // through L1, leaving the shared memory to the weight stages.
  a.act_smem = ROWS || K * 2 <= kActSmemMax ? 1 : 0;
  const int act_bytes = a.act_smem ? a.M * K * 2 : 0;
  const int avail = (ROWS ? kTwoBudgetRows : kTwoBudget) - act_bytes - rps_two - 1024;
  for (int mult = 1; mult <= 2 && cps == 0; ++mult) {
    const int g = ctx.num_sms * mult < a.ntiles ? ctx.num_sms * mult : a.ntiles;
    const int max_tiles = (a.ntiles + g - 1) / g;
    for (int want = 3; want >= 2 && cps == 0 && avail > 0; --want) {
      const int target = avail / want - rps_two < kStageTargetTwo ? avail / want - rps_two : kStageTargetTwo;
      if (!choose(target)) continue;
      const int need = max_tiles * NWT * a.nslices;  // stages of the busiest CTA
      int stages = avail / (a.stage_bytes + rps_two);
      if (stages > kMaxStages) stages = kMaxStages;
      if (stages > need) stages = need;
      const bool all_fit = stages >= 1 && stages == need;
      if ((mult == 1 && all_fit) || (mult == 2 && stages >= 2 && a.stage_bytes >= kTwoMinStage)) {
        cps = 2;
        grid = g;
        a.stages = stages;
      }
    }
  }
  if (ROWS && (cps != 2 || a.stages < (a.ntiles + grid - 1) / grid * a.nslices))
    return cudaErrorNotSupported;  // the row mapping needs every tile of a CTA in flight
  if (cps == 0) {
    cps = 1;
    grid = ctx.num_sms < a.ntiles ? ctx.num_sms : a.ntiles;
    if (!choose(kStageTargetOne)) return cudaErrorNotSupported;
    a.stages = (kOneBudget - act_bytes - rps_one - 1024) / (a.stage_bytes + rps_one);
    if (a.stages > kMaxStages) a.stages = kMaxStages;
    if (a.stages < 2) return cudaErrorNotSupported;
  }
  const bool two = cps > 1;
  const int ncw = two ? kNcwTwo : kNcwOne;
  a.red_off = a.stages * a.stage_bytes + act_bytes;
  const size_t smem = (size_t)a.red_off + (size_t)(a.stages + 1) * NWT * ncw * red_per_warp<PAIR>() * 4 + 1024;
  a.status = ctx.status;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = PAIR ? 0 : ctx.bias_mode;

  // Tensor maps: packed bytes as [K/256 segments][N rows][128 bytes] (box 128 x 16 x nseg)
  // and scales as [srow/128][N][128] (box 128 x 16 x nsbox) when the scale rows are whole
  // 128 bytes, else [N][srow] (box 128 x 16 per copy, the row tail read as zeros).
  a.s3d = srow % 128 == 0 ? 1 : 0;
  CUtensorMap tp[2], ts[2];
  for (int t = 0; t < 2; ++t) {
    memset(&tp[t], 0, sizeof(CUtensorMap));
    memset(&ts[t], 0, sizeof(CUtensorMap));
    const QWeight& q = w[t < NWT ? t : 0];
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t pdim[3] = {128, (cuuint64_t)N, (cuuint64_t)(K / kBlockK)};
    const cuuint64_t pstride[2] = {(cuuint64_t)(K / 2), 128};
    const cuuint32_t pbox[3] = {128, (cuuint32_t)kRows, (cuuint32_t)a.nseg};
    if (encode(&tp[t], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(q.packed), pdim, pstride, pbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
    CUresult r;
    if (a.s3d) {
      const cuuint64_t sdim[3] = {128, (cuuint64_t)N, (cuuint64_t)(srow / 128)};
      const cuuint64_t sstride[2] = {(cuuint64_t)srow, 128};
      const cuuint32_t sbox[3] = {128, (cuuint32_t)kRows, (cuuint32_t)a.nsbox};
      r = encode(&ts[t], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(q.scales), sdim, sstride, sbox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      const cuuint64_t sdim[2] = {(cuuint64_t)srow, (cuuint64_t)N};
      const cuuint64_t sstride[1] = {(cuuint64_t)srow};
      const cuuint32_t sbox[2] = {128, (cuuint32_t)kRows};
      r = encode(&ts[t], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(q.scales), sdim, sstride, sbox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return cudaErrorNotSupported;
  }
  const int cpg = bs / 32;
  MmaKernel kern = nullptr;
  if (ROWS) {
    kern = pick_rows(s16, zp, cpg);
  } else {
    if (cps == 2) kern = a.act_smem ? pick<2, PAIR, true>(s16, zp, cpg) : pick<2, PAIR, false>(s16, zp, cpg);
    if (cps == 1) kern = a.act_smem ? pick<1, PAIR, true>(s16, zp, cpg) : pick<1, PAIR, false>(s16, zp, cpg);
  }
  if (kern == nullptr) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ctx.variant = PAIR ? "gemv_pair_swiglu_mma" : (ROWS ? "gemm_rows_mma" : "gemv_mma");
  const int threads = (ncw + 1) * 32;
  return launch_kernel(ctx, kern, dim3(grid), dim3(threads), smem, a, tp[0], tp[1], ts[0], ts[1]);
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

cudaError_t launch_gemm_rows_mma(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N, int bs,
                                 void* Y) {
  return launch_mma_impl<false, true>(ctx, A, &w, K, N, bs, Y, M);
}

}  // namespace mnb
