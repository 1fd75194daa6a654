// Speculative-verify GEMM, 2 <= M <= 16: Y[M,N] = A[M,K] . dequant(B)^T.
//
// HBM-bound (each weight is used M <= 16 times), so every weight byte is read once and
// the dequantised values never touch shared memory: a CTA owns tiles of 16 weight rows,
// a producer warp streams each tile into a shared-memory ring (packed rows by one bulk
// copy per row, with a 16-byte row pad so the fragment loads are bank-conflict free;
// scales as 128-byte-swizzled 2-D tensor boxes, or one bulk copy per row when a slice's
// scales are not whole boxes; zero points as one copy), and sixteen consumer warps in two
// groups of eight work on two tiles at once, the eight warps of a group splitting K.  A
// lane converts one 32-bit word (8 nibbles) of row g and of row g+8 into exact fp16
// (code - zp) and feeds them to two mma.sync.m16n8k16 (fp32 accumulate) as the A
// operand; the activations, staged once per CTA, are the B operand (8 rows of A per
// instruction, two instructions per step for M > 8).
//
// The k index inside each MMA is permuted the same way for both operands: lane
// (g, t) supplies physical k = 8t + {0,4,1,5} to the first MMA and 8t + {2,6,3,7} to the
// second, which is exactly the pairing the magic-number conversion produces, so no
// register shuffles are needed.  Each MMA spans one 32-k chunk, inside one quant group
// for block sizes >= 32.  A warp walks its K range group by group (1, 2 or 4 chunks per
// group, a template parameter): it reads the group's scale and zero point of its two rows
// once, accumulates the group's MMAs into a fresh fp32 fragment and adds that fragment
// times the group scale to the running sum (scale after accumulate, as in
// matmul_nbits_marlin_gemm_f16 of marlin_gemm.rs).  The eight scale rows a warp reads
// together sit in eight banks (swizzled boxes, or row-copied rows at a stride of 16 mod
// 32 bytes), and lanes whose activation row is past M skip their activation reads.  Block
// size 16 puts two groups in a chunk (see the CPG == 0 branch).
#include <cuda.h>
#include <cstring>
#include <cudaTypedefs.h>

#include "mma_sync.cuh"
#include "mnb_device.cuh"
#include "mnb_internal.h"
#include "tcgen05.cuh"

namespace mnb {
namespace {

constexpr int kRows = 16;        // weight rows per tile
constexpr int kCW = 16;          // consumer warps
constexpr int kGroups = 2;       // tiles worked on at once (8 warps each)
constexpr int kGW = kCW / kGroups;
constexpr int kThreads = (kCW + 1) * 32;
constexpr int kRowPad = 16;      // bytes between staged rows
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 208 * 1024;  // dynamic; static shared memory is at most ~17 KB

struct SmArgs {
  const __half* A;
  const uint8_t* packed;
  const uint8_t* scales;
  const uint8_t* zp;
  __half* Y;
  int M, K, N, G, gshift;
  int row_bytes;     // K / 2 (packed row stride in global memory)
  int srow;          // scale bytes per row in global memory
  int ssz;           // bytes per scale
  int zrow;          // zero-point bytes per row (0 if none); staged whole
  // Split-K: grid.y = nslices slices of kslice k (the last one shorter); a slice stages its
  // packed codes and scales, and with more than one slice writes fp32 partials to
  // part[slice][m][n], which combine_slices_kernel adds in slice order.
  int kslice, nslices;
  float* part;
  int sslice;        // scale bytes per row of a slice (kslice / bs * ssz)
  int sstride;       // staged scale row stride: sslice rounded up to 16 mod 32 bytes, so the
                     // eight rows a warp reads for one group fall in eight different banks
  int prow;          // staged row stride = kslice / 2 + kRowPad
  int stage_bytes;   // one ring slot (a multiple of 1024 with tensor-copied scales)
  // Stage layout: packed rows at poff, scales at soff, zero points at zoff.  With stma the
  // scales arrive as nsb 2-D tensor copies of 16 rows x 128 bytes each (128-byte
  // swizzle, 1024-aligned): byte b of row r of box i sits at i * 2048 + r * 128 +
  // (b ^ 16 (r mod 8)); otherwise as one copy per row at stride sstride.
  int stma, nsb;
  int poff, soff, zoff;
  int stages;
  int xstride;       // two row sets: staged activation row stride (bytes)
  int ntiles, tiles_per_cta;
  uint32_t* status;
  const __half* bias;
  int bias_mode;
  // fp32 output (F32): A holds 2 * Mout rows, row 2m = hi and row 2m + 1 = lo of fp32 row m
  // scaled by 2^-rexp[m]; Yf[m, n] = 2^rexp[m] * (y[2m, n] + y[2m + 1, n]) + biasf[n].
  int Mout;
  float* Yf;
  const float* biasf;
  const int* rexp;
};

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCW * 32) : "memory");
}
__device__ __forceinline__ void group_bar(int gi) {
  asm volatile("bar.sync %0, %1;" ::"r"(2 + gi), "n"(kGW * 32) : "memory");
}

// Fixed-order sum over the K slices of the staged partials of activation row m, weight row
// `row` of the tile.
template <int MSETS>
__device__ __forceinline__ float slice_sum(const float (&red)[kGW][MSETS][32][4], int row, int m) {
  const int s = m >> 3, mm = m & 7;
  const int l = (row & 7) * 4 + (mm >> 1), j = ((row >> 3) << 1) + (mm & 1);
  float v = 0.0f;
#pragma unroll
  for (int w = 0; w < kGW; ++w) v += red[w][s][l][j];
  return v;
}

// CPG: 32-k chunks per quant group (block size 32, 64 or 128).  The scale dtype is a
// runtime property (one uniform branch per group); zero points are a template flag.
//
// Two row sets (M > 8) stage the activation rows by one bulk copy per row (row stride 64
// mod 128 bytes, so the two rows a quarter-warp reads sit in different banks); lanes pair
// the halves after loading them.  One row set stages the fragment order, with plain loads.
template <int MSETS, int CPG, bool ZP, bool F32 = false, bool SPLIT = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_smallm_kernel(const SmArgs p, const __grid_constant__ CUtensorMap tmap_s) {
  constexpr bool kTwoSets = MSETS == 2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ uint64_t x_bar;
  __shared__ __align__(16) float red[kGroups][kGW][MSETS][32][4];  // float4 stores
  __shared__ int failed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = SPLIT ? (int)blockIdx.y : 0;
  const int k0 = SPLIT ? slice * p.kslice : 0;     // first k of this slice
  const int klen = SPLIT ? min(p.kslice, p.K - k0) : p.K;
  const int C = klen >> 5;                         // 32-k chunks in the slice
  const int gb = SPLIT ? (k0 >> p.gshift) : 0;     // first group of the slice
  const int S = p.stages;
  // shared memory: [ring stages][activations: fragment order (one row set) or rows (two sets)]
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned slots
  uint8_t* xs = ring + (size_t)S * p.stage_bytes;
  const int t_begin = blockIdx.x * p.tiles_per_cta;
  const int t_end = min(p.ntiles, t_begin + p.tiles_per_cta);
  const int ntile = max(0, t_end - t_begin);

  if (tid == 0) {
    failed = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kGW);
    }
    if (kTwoSets) mbar_init(&x_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool x_issued = false, x_ok = true;

  if (warp == kCW) {
    // ------------------------------ producer ------------------------------------
    // Lane 0 waits for the slot and arms its barrier; then lane r issues row r's copies,
    // so a tile's row copies go out as one warp instruction each.
    int slot = 0, issued = 0;
    uint32_t phase = 0;
    for (int i = 0; i < ntile; ++i) {
      int free_slot = 1;
      if (lane == 0 && issued >= S && !mbar_wait_bounded(&empty_bar[slot], phase ^ 1u)) {
        report_status(p.status, kStatusEmptyWait);
        atomicExch(&failed, 1);
        free_slot = 0;
      }
      if (!__shfl_sync(0xffffffffu, free_slot, 0)) break;
      const int n0 = (t_begin + i) * kRows;
      const int nr = min(kRows, p.N - n0);
      uint8_t* st = ring + (size_t)slot * p.stage_bytes;
      const int pbytes = klen >> 1, sbytes = (klen >> p.gshift) * p.ssz;
      // A tensor box always lands (and counts) whole: 16 rows x 128 bytes, rows past N zero.
      const int nboxes = sbytes >> 7;
      const uint32_t bytes = (uint32_t)nr * (pbytes + p.zrow) + (p.stma ? (uint32_t)nboxes * 2048u : (uint32_t)(nr * sbytes));
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[slot], bytes);
      __syncwarp();
      if (lane < nr)
        bulk_g2s(st + p.poff + lane * p.prow, p.packed + (long long)(n0 + lane) * p.row_bytes + (k0 >> 1), pbytes,
                 &full_bar[slot]);
      if (p.stma) {
        if (lane == 1)
          for (int b = 0; b < nboxes; ++b)
            tc::tma_load_2d(st + p.soff + b * 2048, &tmap_s, gb * p.ssz + b * 128, n0, &full_bar[slot]);
      } else if (lane < nr) {
        bulk_g2s(st + p.soff + lane * p.sstride, p.scales + (long long)(n0 + lane) * p.srow + gb * p.ssz, sbytes,
                 &full_bar[slot]);
      }
      if (ZP && lane == 0)
        bulk_g2s(st + p.zoff, p.zp + (long long)n0 * p.zrow, nr * p.zrow, &full_bar[slot]);
      ++issued;
      if (++slot == S) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (lane == 0)
      for (int i = issued > S ? issued - S : 0; i < issued; ++i)
        (void)mbar_wait_bounded(&full_bar[i % S], (uint32_t)(i / S) & 1u);
    pdl_launch_dependents();
  } else {
    // ------------------------------ consumers -----------------------------------
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t xs_u32 = smem_u32(xs);
    if constexpr (kTwoSets) {
      // One lane copies every activation row of the slice into this CTA's shared memory.
      if (warp == 0 && lane == 0) {
        mbar_arrive_expect_tx(&x_bar, (uint32_t)(p.M * klen * 2));
        for (int m = 0; m < p.M; ++m)
          bulk_g2s(xs + (size_t)m * p.xstride, p.A + (long long)m * p.K + k0, (uint32_t)(klen * 2), &x_bar);
        x_issued = true;
      }
      if (!mbar_wait_bounded(&x_bar, 0)) {
        report_status(p.status, kStatusFullWait);
        atomicExch(&failed, 1);
        x_ok = false;
      }
    } else {
      // Stage the activations once, compactly: entry (chunk c, row m < M, quarter t) holds
      // A[m][k0 + 32c + 8t .. +8], paired (x0,x4)(x1,x5)(x2,x6)(x3,x7), at byte
      // ((c M + m) 4 + t) 16, so lane 4g + t finds row g of chunk c at 16 lane + 64 M c.
      // Thread i fills quarter-chunks j = i, i + 512, ... of every row, all rows' loads in
      // flight before the first store.
      {
        const int J = 4 * C;  // quarter-chunks (8 halves) per row
        for (int j = tid; j < J; j += kCW * 32) {
          uint4 x[8];
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            x[m] = make_uint4(0, 0, 0, 0);
            if (m < p.M) x[m] = *reinterpret_cast<const uint4*>(p.A + (long long)m * p.K + k0 + 8 * j);
          }
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            if (m < p.M) {
              uint32_t q[4];
              pair_halves_stride4(x[m], q);
              asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                               xs_u32 + (uint32_t)((((j >> 2) * p.M + m) * 4 + (j & 3)) * 16)),
                           "r"(q[0]), "r"(q[1]), "r"(q[2]), "r"(q[3])
                           : "memory");
            }
          }
        }
      }
      consumer_bar();
    }

    const int g = lane >> 2, t = lane & 3;
    const int gi = warp / kGW, gw = warp % kGW;  // tile group, warp within it
    const int Gs = CPG > 0 ? C / CPG : 2 * C;   // quant groups in the slice
    const int q_lo = (gw * Gs) / kGW, q_hi = ((gw + 1) * Gs) / kGW;  // this warp's groups
    const bool s16 = p.ssz == 2;
    const uint32_t zl8 = zp_lo_const(8u), zh8 = zp_hi_const(8u);
    // One row set: this lane's activation fragment of chunk c sits at 16 lane + 64 M c.
    // Lanes whose activation row is past M hold zeros and skip the shared-memory read.
    const uint32_t xlane = xs_u32 + (uint32_t)lane * 16u;
    const uint32_t xcstride = 64u * (uint32_t)p.M;
    bool xlive[MSETS];
    uint32_t xrow[MSETS];  // two-set layout: this lane's 16 bytes of row 8s + g, chunk 0
#pragma unroll
    for (int s = 0; s < MSETS; ++s) {
      xlive[s] = 8 * s + g < p.M;
      xrow[s] = xs_u32 + (uint32_t)((8 * s + g) * p.xstride) + 16u * (uint32_t)t;
    }
    bool ok = x_ok;
    for (int i = gi; i < ntile; i += kGroups) {
      const int slot = i % S;
      const uint32_t phase = (uint32_t)(i / S) & 1u;
      if (ok && !mbar_wait_bounded(&full_bar[slot], phase)) {
        report_status(p.status, kStatusFullWait);
        atomicExch(&failed, 1);
        ok = false;
      }
      const uint32_t st = smem_u32(ring + (size_t)slot * p.stage_bytes);
      const uint32_t rowg = st + (uint32_t)(p.poff + g * p.prow) + 4u * t;
      const uint32_t rowg8 = rowg + (uint32_t)(8 * p.prow);
      const uint32_t sbase = st + (uint32_t)p.soff;
      const uint32_t sg_row = sbase + (uint32_t)(g * p.sstride);  // row-copied scales
      // Shared-memory address of byte `off` of this lane's scale row g (row g + 8: + hi8).
      const uint32_t hi8 = p.stma ? 1024u : (uint32_t)(8 * p.sstride);
      auto scale_addr = [&](uint32_t off) -> uint32_t {
        return p.stma ? sbase + (off >> 7) * 2048u + (uint32_t)g * 128u + ((off & 127u) ^ ((uint32_t)g << 4))
                      : sg_row + off;
      };
      const uint32_t zg_row = st + (uint32_t)(p.zoff + g * p.zrow);
      const uint32_t zg8_row = zg_row + (uint32_t)(8 * p.zrow);
      float acc[MSETS][4];
#pragma unroll
      for (int s = 0; s < MSETS; ++s)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[s][j] = 0.0f;
      if constexpr (CPG == 0) {
      if (ok) {
        // Block size 16: chunk c holds groups 2c (the words of lanes t < 2) and 2c + 1
        // (t >= 2).  Each lane converts with its own group's zero point; each MMA step runs
        // twice with the activation fragment of the other group's lanes zeroed, so the
        // two groups accumulate into separate fragments, each scaled after accumulation.
        const bool lo_half = t < 2;
        const int c_lo = (gw * C) / kGW, c_hi = ((gw + 1) * C) / kGW;
        for (int c = c_lo; c < c_hi; ++c) {
          float sa, sa8, sb, sb8;  // scales of groups 2c (a) and 2c + 1 (b), rows g and g + 8
          if (s16) {
            const uint32_t sa_ = scale_addr(4u * (uint32_t)c);
            const uint32_t h = lds_u32_a(sa_), h8 = lds_u32_a(sa_ + hi8);
            sa = half_bits_to_float(h & 0xffffu);
            sb = half_bits_to_float(h >> 16);
            sa8 = half_bits_to_float(h8 & 0xffffu);
            sb8 = half_bits_to_float(h8 >> 16);
          } else {
            const uint32_t sa_ = scale_addr(8u * (uint32_t)c);
            const uint2 f = lds_u64_a(sa_), f8 = lds_u64_a(sa_ + hi8);
            sa = __uint_as_float(f.x);
            sb = __uint_as_float(f.y);
            sa8 = __uint_as_float(f8.x);
            sb8 = __uint_as_float(f8.y);
          }
          uint32_t zl = zl8, zh = zh8, zl_8 = zl8, zh_8 = zh8;
          if (ZP) {
            // zero-point byte (gb + 2c) / 2 holds group 2c (low nibble) and 2c + 1 (high)
            const uint32_t zb = (uint32_t)((gb >> 1) + c);
            const uint32_t b0 = lds_u8_a(zg_row + zb), b1 = lds_u8_a(zg8_row + zb);
            const uint32_t z0 = lo_half ? (b0 & 15u) : (b0 >> 4), z1 = lo_half ? (b1 & 15u) : (b1 >> 4);
            zl = zp_lo_const(z0);
            zh = zp_hi_const(z0);
            zl_8 = zp_lo_const(z1);
            zh_8 = zp_hi_const(z1);
          }
          const uint32_t wa = lds_u32_a(rowg + 16u * (uint32_t)c);
          const uint32_t wb = lds_u32_a(rowg8 + 16u * (uint32_t)c);
          uint32_t da[4], db[4];
          nibbles_to_centered_half2(wa, zl, zh, da);
          nibbles_to_centered_half2(wb, zl_8, zh_8, db);
#pragma unroll
          for (int s = 0; s < MSETS; ++s) {
            uint4 xf = make_uint4(0, 0, 0, 0);
            if (xlive[s]) {
              if constexpr (kTwoSets) {
                uint32_t q[4];
                pair_halves_stride4(lds128_a(xrow[s] + 64u * (uint32_t)c), q);
                xf = make_uint4(q[0], q[1], q[2], q[3]);
              } else {
                xf = lds128_a(xlane + (uint32_t)c * xcstride);
              }
            }
            const uint4 xa = lo_half ? xf : make_uint4(0, 0, 0, 0);
            const uint4 xb = lo_half ? make_uint4(0, 0, 0, 0) : xf;
            float ta[4], tb[4];
            mma16816_zero(ta, da[0], db[0], da[1], db[1], xa.x, xa.y);
            mma16816(ta, da[2], db[2], da[3], db[3], xa.z, xa.w);
            mma16816_zero(tb, da[0], db[0], da[1], db[1], xb.x, xb.y);
            mma16816(tb, da[2], db[2], da[3], db[3], xb.z, xb.w);
            acc[s][0] = fmaf(tb[0], sb, fmaf(ta[0], sa, acc[s][0]));
            acc[s][1] = fmaf(tb[1], sb, fmaf(ta[1], sa, acc[s][1]));
            acc[s][2] = fmaf(tb[2], sb8, fmaf(ta[2], sa8, acc[s][2]));
            acc[s][3] = fmaf(tb[3], sb8, fmaf(ta[3], sa8, acc[s][3]));
          }
        }
      }
      } else if (ok) {
        for (int q = q_lo; q < q_hi; ++q) {
          // Group q of the slice: its scales (rows g and g + 8) and zero points.
          float sg, sg8;
          if (s16) {
            const uint32_t sa_ = scale_addr(2u * (uint32_t)q);
            sg = half_bits_to_float(lds_u16_a(sa_));
            sg8 = half_bits_to_float(lds_u16_a(sa_ + hi8));
          } else {
            const uint32_t sa_ = scale_addr(4u * (uint32_t)q);
            sg = __uint_as_float(lds_u32_a(sa_));
            sg8 = __uint_as_float(lds_u32_a(sa_ + hi8));
          }
          uint32_t zlg = zl8, zhg = zh8, zlg8 = zl8, zhg8 = zh8;
          if (ZP) {
            const int grp = gb + q;  // zero points are staged as whole rows
            const uint32_t sh = (uint32_t)(grp & 1) * 4u;
            const uint32_t z0 = (lds_u8_a(zg_row + (uint32_t)(grp >> 1)) >> sh) & 15u;
            const uint32_t z1 = (lds_u8_a(zg8_row + (uint32_t)(grp >> 1)) >> sh) & 15u;
            zlg = zp_lo_const(z0);
            zhg = zp_hi_const(z0);
            zlg8 = zp_lo_const(z1);
            zhg8 = zp_hi_const(z1);
          }
          // Fresh fp32 fragments for the group: chain 1 takes physical k = 8t + {0,4,1,5},
          // chain 2 k = 8t + {2,6,3,7} of each chunk (one chain for single-chunk groups).
          float tmp[MSETS][4], tmp2[MSETS][4];
#pragma unroll
          for (int cc = 0; cc < CPG; ++cc) {
            const uint32_t c = (uint32_t)(q * CPG + cc);
            const uint32_t wa = lds_u32_a(rowg + 16u * c);
            const uint32_t wb = lds_u32_a(rowg8 + 16u * c);
            uint32_t da[4], db[4];
            nibbles_to_centered_half2(wa, zlg, zhg, da);
            nibbles_to_centered_half2(wb, zlg8, zhg8, db);
#pragma unroll
            for (int s = 0; s < MSETS; ++s) {
              uint4 xf = make_uint4(0, 0, 0, 0);
              if (xlive[s]) {
                if constexpr (kTwoSets) {
                  uint32_t q[4];
                  pair_halves_stride4(lds128_a(xrow[s] + 64u * c), q);
                  xf = make_uint4(q[0], q[1], q[2], q[3]);
                } else {
                  xf = lds128_a(xlane + c * xcstride);
                }
              }
              if (CPG == 1) {
                mma16816_zero(tmp[s], da[0], db[0], da[1], db[1], xf.x, xf.y);
                mma16816(tmp[s], da[2], db[2], da[3], db[3], xf.z, xf.w);
              } else if (cc == 0) {
                mma16816_zero(tmp[s], da[0], db[0], da[1], db[1], xf.x, xf.y);
                mma16816_zero(tmp2[s], da[2], db[2], da[3], db[3], xf.z, xf.w);
              } else {
                mma16816(tmp[s], da[0], db[0], da[1], db[1], xf.x, xf.y);
                mma16816(tmp2[s], da[2], db[2], da[3], db[3], xf.z, xf.w);
              }
            }
          }
#pragma unroll
          for (int s = 0; s < MSETS; ++s) {
            if (CPG > 1) {
#pragma unroll
              for (int j = 0; j < 4; ++j) tmp[s][j] += tmp2[s][j];
            }
            acc[s][0] = fmaf(tmp[s][0], sg, acc[s][0]);
            acc[s][1] = fmaf(tmp[s][1], sg, acc[s][1]);
            acc[s][2] = fmaf(tmp[s][2], sg8, acc[s][2]);
            acc[s][3] = fmaf(tmp[s][3], sg8, acc[s][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
#pragma unroll
      for (int s = 0; s < MSETS; ++s)
        *reinterpret_cast<float4*>(&red[gi][gw][s][lane][0]) = make_float4(acc[s][0], acc[s][1], acc[s][2], acc[s][3]);
      group_bar(gi);
      // Fixed-order sum over the warps' K ranges; one thread per (row, m).
      const int n0 = (t_begin + i) * kRows;
      if constexpr (F32) {
        for (int e = gw * 32 + lane; e < kRows * p.Mout; e += kGW * 32) {
          const int row = e % kRows, m = e / kRows;
          const float v = slice_sum<MSETS>(red[gi], row, 2 * m) + slice_sum<MSETS>(red[gi], row, 2 * m + 1);
          const int n = n0 + row;
          if (n < p.N) {
            p.Yf[(long long)m * p.N + n] =
                failed ? __uint_as_float(0x7fc00000u) : ldexpf(v, p.rexp[m]) + (p.biasf ? p.biasf[n] : 0.0f);
          }
        }
      } else {
        for (int e = gw * 32 + lane; e < kRows * 8 * MSETS; e += kGW * 32) {
          const int row = e % kRows, m = e / kRows;
          const float v = slice_sum<MSETS>(red[gi], row, m);
          const int n = n0 + row;
          if (m < p.M && n < p.N) {
            if constexpr (SPLIT)
              p.part[((long long)slice * p.M + m) * p.N + n] = failed ? __uint_as_float(0x7fc00000u) : v;
            else
              p.Y[(long long)m * p.N + n] = failed ? __ushort_as_half(0x7e00) : round_out(v, p.bias, n, p.bias_mode);
          }
        }
      }
      group_bar(gi);
    }
  }
  if constexpr (kTwoSets) {
    // The CTA does not leave while an activation copy it issued may still land.
    if (x_issued && !x_ok) (void)mbar_wait_bounded(&x_bar, 0);
  }
}

// Fixed-order sum of the split-K partials, then the fp16 epilogue (bias modes).
__global__ void __launch_bounds__(256) combine_slices_kernel(const float* __restrict__ part, int nslices,
                                                             long long mn, int N, __half* __restrict__ Y,
                                                             const __half* bias, int bias_mode) {
  pdl_launch_dependents();
  pdl_wait();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < mn; i += (long long)gridDim.x * blockDim.x) {
    float v = 0.0f;
    for (int s = 0; s < nslices; ++s) v += part[s * mn + i];
    Y[i] = round_out(v, bias, (int)(i % N), bias_mode);
  }
}

// fp32 output of split activations, summed over the K slices in slice order:
// Yf[m, n] = 2^rexp[m] * sum_s (part[s][2m][n] + part[s][2m + 1][n]) + biasf[n].
__global__ void __launch_bounds__(256) combine_slices_f32_kernel(const float* __restrict__ part, int nslices,
                                                                 int Mout, int N, float* __restrict__ Yf,
                                                                 const float* biasf, const int* rexp) {
  pdl_launch_dependents();
  pdl_wait();
  const long long mn = (long long)Mout * N, rows = 2LL * Mout * N;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < mn; i += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(i / N), n = (int)(i % N);
    float v = 0.0f;
    for (int s = 0; s < nslices; ++s) {
      const float* ps = part + s * rows + (long long)(2 * m) * N + n;
      v += ps[0] + ps[N];
    }
    Yf[i] = ldexpf(v, rexp[m]) + (biasf ? biasf[n] : 0.0f);
  }
}

using SmKernel = void (*)(const SmArgs, const CUtensorMap);

template <int MSETS, int CPG, bool F32, bool SPLIT>
SmKernel pick_zp(bool zp) {
  return zp ? gemm_smallm_kernel<MSETS, CPG, true, F32, SPLIT> : gemm_smallm_kernel<MSETS, CPG, false, F32, SPLIT>;
}

// cpg: 32-k chunks per quant group (1, 2 or 4; 0 for block size 16, two groups per
// chunk); anything else is not handled.
template <int MSETS, bool F32, bool SPLIT = false>
SmKernel pick(int cpg, bool zp) {
  if (cpg == 0) return pick_zp<MSETS, 0, F32, SPLIT>(zp);
  if (cpg == 1) return pick_zp<MSETS, 1, F32, SPLIT>(zp);
  if (cpg == 2) return pick_zp<MSETS, 2, F32, SPLIT>(zp);
  if (cpg == 4) return pick_zp<MSETS, 4, F32, SPLIT>(zp);
  return nullptr;
}

}  // namespace

// Staged scale row stride for `bytes` of scales per row (a multiple of 16): congruent to 16
// mod 32 bytes, so row r starts at bank 4 * (r * odd mod 8) and eight rows never collide.
static int scale_stride(int bytes) { return bytes % 32 == 0 ? bytes + 16 : bytes; }

// Activation row stride of the two-row-set layout for a slice of ks k (2 * ks is a multiple of
// 64): congruent to 64 mod 128 bytes.
static int two_set_x_stride(int ks) { return (2 * ks) % 128 == 0 ? 2 * ks + 64 : 2 * ks; }

// Shared memory for the staged activations of a slice of ks k.
static size_t x_bytes(int M, int ks) {
  if (M <= 8) return (size_t)2 * M * ks;  // one row set, compact fragment order
  return (size_t)M * two_set_x_stride(ks);
}

// K-slice length for the small-M kernel: all of K when its rows, scales and activations fit
// two ring slots, else the largest of 4096 / 2048 / 1024 (multiples of the block size) that
// fits.  ssz: bytes per scale; zp: zero points present.  0: not handled.
int smallm_kslice(int M, int K, int bs, int ssz, bool zp) {
  if (M < 2 || M > 16 || bs < 16 || K % 32 != 0) return 0;
  const int G = K / bs, zrow = zp ? (G + 1) / 2 : 0;
  auto fits = [&](int ks) {
    // two ring slots (either scale layout, 1024-aligned) + activations + base alignment
    const size_t stage = ((size_t)kRows * (ks / 2 + kRowPad + scale_stride((ks / bs) * ssz) + zrow) + 1023) / 1024 * 1024;
    return x_bytes(M, ks) + 2 * stage + 1024 <= (size_t)kSmemBudget;
  };
  if (fits(K)) return K;
  for (int ks : {4096, 2048, 1024})
    if (ks < K && ks % bs == 0 && fits(ks)) return ks;
  return 0;
}

// Upper bound over the scale dtype and zero points: the slicing with fp32 scales and zero
// points (the largest footprint, hence the most slices) needs the most partials.
size_t smallm_workspace_bytes(int M, int K, int N, int bs) {
  const int ks = smallm_kslice(M, K, bs, 4, true);
  if (ks == 0 || ks >= K) return 0;
  const size_t ns = (size_t)((K + ks - 1) / ks);
  return ns * (size_t)M * (size_t)N * 4;
}

namespace {

cudaError_t launch_smallm_impl(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N, int bs,
                               void* Y, int Mout, float* Yf, const float* biasf, const int* rexp,
                               void* workspace = nullptr, size_t ws_bytes = 0) {
  if (M < 2 || M > 16 || (bs != 16 && bs != 32 && bs != 64 && bs != 128) || K % 32 != 0)
    return cudaErrorNotSupported;
  SmArgs a = {};
  a.A = static_cast<const __half*>(A);
  a.packed = w.packed;
  a.scales = static_cast<const uint8_t*>(w.scales);
  a.zp = w.zp;
  a.Y = static_cast<__half*>(Y);
  a.M = M;
  a.K = K;
  a.N = N;
  a.G = K / bs;
  a.gshift = 0;
  while ((1 << a.gshift) < bs) ++a.gshift;
  a.row_bytes = K / 2;
  a.ssz = w.scales_f16 ? 2 : 4;
  a.srow = a.G * a.ssz;
  a.zrow = w.zp ? (a.G + 1) / 2 : 0;
  const int ks = smallm_kslice(M, K, bs, a.ssz, w.zp != nullptr);
  if (ks == 0) return cudaErrorNotSupported;
  a.kslice = ks;
  a.nslices = (K + ks - 1) / ks;
  const int klast = K - (a.nslices - 1) * ks;
  a.sslice = (ks / bs) * a.ssz;
  a.sstride = scale_stride(a.sslice);
  // Every bulk copy is a 16-byte multiple at a 16-byte offset: packed slices (k multiples
  // of 32), scale slices (checked here, also the last one, and the row stride) and a tile's
  // zero-point rows (16 * zrow bytes at a multiple of 16 * zrow: any zrow works for whole
  // tiles; a partial last tile needs zrow itself to be a multiple of 16).
  if (a.sslice % 16 != 0 || ((klast / bs) * a.ssz) % 16 != 0 || a.srow % 16 != 0 ||
      (a.zrow % 16 != 0 && N % kRows != 0))
    return cudaErrorNotSupported;
  if (a.nslices > 1) {
    // More than one slice needs the partials workspace (for fp32 output: partials of the
    // 2 * Mout split rows, combined with their exponents afterwards).
    if (workspace == nullptr || ws_bytes < (size_t)a.nslices * M * N * 4) return cudaErrorNotSupported;
    a.part = static_cast<float*>(workspace);
  }
  a.prow = ks / 2 + kRowPad;
  // Scales by 128-byte tensor boxes when every slice's scale bytes are whole boxes (one
  // copy per 2 KB instead of one per row), else one bulk copy per row.
  CUtensorMap tmap_s;
  memset(&tmap_s, 0, sizeof(tmap_s));
  a.stma = 0;
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (encode && a.sslice % 128 == 0 && ((klast / bs) * a.ssz) % 128 == 0) {
    const cuuint64_t gdim[2] = {(cuuint64_t)a.srow, (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)a.srow};
    const cuuint32_t box[2] = {128, (cuuint32_t)kRows};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmap_s, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(w.scales), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      a.stma = 1;
  }
  if (a.stma) {
    a.nsb = a.sslice / 128;
    a.soff = 0;
    a.poff = a.nsb * 2048;
    a.zoff = a.poff + kRows * a.prow;
    a.stage_bytes = (a.zoff + kRows * a.zrow + 1023) / 1024 * 1024;
  } else {
    a.nsb = 0;
    a.poff = 0;
    a.soff = kRows * a.prow;
    a.zoff = a.soff + kRows * a.sstride;
    a.stage_bytes = a.zoff + kRows * a.zrow;
  }
  const int msets = M <= 8 ? 1 : 2;
  const size_t xbytes = x_bytes(M, ks);
  a.xstride = two_set_x_stride(ks);
  const size_t usable = (size_t)kSmemBudget - 1024;  // minus the base-alignment slack
  if (usable < xbytes + 2 * (size_t)a.stage_bytes) return cudaErrorNotSupported;
  a.stages = (int)((usable - xbytes) / a.stage_bytes);
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  a.ntiles = (N + kRows - 1) / kRows;
  // Spread (tile, slice) units over the SMs: each slice gets num_sms / nslices CTAs.
  const int ctas_per_slice = ctx.num_sms / a.nslices > 0 ? ctx.num_sms / a.nslices : 1;
  a.tiles_per_cta = (a.ntiles + ctas_per_slice - 1) / ctas_per_slice;
  int grid = (a.ntiles + a.tiles_per_cta - 1) / a.tiles_per_cta;
  a.status = ctx.status;
  a.bias = static_cast<const __half*>(ctx.bias);
  a.bias_mode = ctx.bias_mode;
  a.Mout = Mout;
  a.Yf = Yf;
  a.biasf = biasf;
  a.rexp = rexp;
  const bool f32 = Yf != nullptr;
  const size_t smem = (size_t)a.stages * a.stage_bytes + xbytes + 1024;
  const bool zp = w.zp != nullptr;
  const int cpg = bs / 32;  // 0 for block size 16
  const bool split = a.nslices > 1;  // split calls write plain partials, fp32 output or not
  SmKernel kern = msets == 1 ? (split ? pick<1, false, true>(cpg, zp) : (f32 ? pick<1, true>(cpg, zp) : pick<1, false>(cpg, zp)))
                             : (split ? pick<2, false, true>(cpg, zp) : (f32 ? pick<2, true>(cpg, zp) : pick<2, false>(cpg, zp)));
  if (kern == nullptr) return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ctx.variant = f32 ? "gemm_smallm_mma16816_f32split" : "gemm_smallm_mma16816";
  auto launch = [&](dim3 g) { return launch_kernel(ctx, kern, g, dim3(kThreads), smem, a, tmap_s); };
  if (a.nslices == 1) return launch(dim3(grid));
  e = launch(dim3(grid, a.nslices));
  if (e != cudaSuccess) return e;
  if (f32) {
    const long long mn = (long long)Mout * N;
    const long long blocks = (mn + 255) / 256, cap = (long long)ctx.num_sms * 8;
    ctx.variant = "gemm_smallm_mma16816_f32split_splitk";
    return launch_kernel(ctx, combine_slices_f32_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0,
                         static_cast<const float*>(a.part), a.nslices, Mout, N, Yf, biasf, rexp);
  }
  const long long mn = (long long)M * N;
  const long long blocks = (mn + 255) / 256, cap = (long long)ctx.num_sms * 8;
  ctx.variant = "gemm_smallm_mma16816_splitk";
  return launch_kernel(ctx, combine_slices_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0,
                       static_cast<const float*>(a.part), a.nslices, mn, N, static_cast<__half*>(Y),
                       static_cast<const __half*>(ctx.bias), ctx.bias_mode);
}

}  // namespace

cudaError_t launch_combine_slices(LaunchCtx& ctx, const float* part, int nslices, int M, int N, void* Y) {
  const long long mn = (long long)M * N;
  const long long blocks = (mn + 255) / 256, cap = (long long)ctx.num_sms * 8;
  return launch_kernel(ctx, combine_slices_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0, part,
                       nslices, mn, N, static_cast<__half*>(Y), static_cast<const __half*>(ctx.bias), ctx.bias_mode);
}

cudaError_t launch_combine_slices_f32(LaunchCtx& ctx, const float* part, int nslices, int Mout, int N, float* Yf,
                                      const float* biasf, const int* rexp) {
  const long long mn = (long long)Mout * N;
  const long long blocks = (mn + 255) / 256, cap = (long long)ctx.num_sms * 8;
  return launch_kernel(ctx, combine_slices_f32_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0,
                       part, nslices, Mout, N, Yf, biasf, rexp);
}

cudaError_t launch_gemm_smallm(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N, int bs,
                               void* Y, void* workspace, size_t ws_bytes) {
  return launch_smallm_impl(ctx, A, M, w, K, N, bs, Y, M, nullptr, nullptr, nullptr, workspace, ws_bytes);
}

cudaError_t launch_gemm_smallm_f32split(LaunchCtx& ctx, const void* A2, int M, const QWeight& w, int K, int N,
                                        int bs, float* Y, const float* bias, const int* rexp, void* workspace,
                                        size_t ws_bytes) {
  if (M < 1 || 2 * M > 16) return cudaErrorNotSupported;
  return launch_smallm_impl(ctx, A2, 2 * M, w, K, N, bs, nullptr, M, Y, bias, rexp, workspace, ws_bytes);
}

}  // namespace mnb
