// Device helpers shared by the mnb kernels (CUDA side only).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace mnb {

constexpr uint32_t kFull = 0xffffffffu;

// ---------------------------------------------------------------------------------
// Programmatic dependent launch.  `pdl_wait` blocks until every kernel this one
// depends on has finished and its writes are visible; before it a kernel may only
// read buffers that no earlier kernel writes (the weights).  Both are no-ops when
// the kernel was launched without programmatic stream serialisation.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 128-bit read-only streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_nc_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_nc_u8(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------------
// Nibbles to exact fp16 (code - zp).
//
// A half whose bit pattern is 0x6400 | x (x < 1024) has the value 1024 + x, so OR-ing a
// nibble into the low mantissa bits of 0x6400 gives 1024 + c, and a nibble sitting four
// bits higher gives 1024 + 16 c.  Subtracting 1024 + zp, or scaling by 1/16 and
// subtracting 64 + zp, leaves c - zp exactly (all values are small integers).  This is
// the bit trick the fp16 GEMV of matmul_nbits.rs builds on; written here with the zero
// point folded into the correction constants.
//
// For a 32-bit word with nibbles n0..n7 (bits 4p..4p+3 hold n_p) the results are the
// half2 pairs (n0,n4), (n1,n5), (n2,n6), (n3,n7), low half first.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(orv));  // (a & b) | c
  return r;
}

// Correction constants for zero point z (0..15): -(1024 + z) and -(64 + z), as half2.
__device__ __forceinline__ uint32_t zp_lo_const(uint32_t z) { return (0xE400u + z) * 0x10001u; }
__device__ __forceinline__ uint32_t zp_hi_const(uint32_t z) { return (0xD400u + 16u * z) * 0x10001u; }

__device__ __forceinline__ void nibbles_to_centered_half2(uint32_t w, uint32_t zlo, uint32_t zhi,
                                                          uint32_t d[4]) {
  const uint32_t kMaskLo = 0x000f000fu, kMaskHi = 0x00f000f0u, kMagic = 0x64006400u;
  const uint32_t kSixteenth = 0x2C002C00u;  // half2(1/16, 1/16)
  const uint32_t t = w >> 8;
  uint32_t h0 = lop3_and_or(w, kMaskLo, kMagic);
  uint32_t h1 = lop3_and_or(w, kMaskHi, kMagic);
  uint32_t h2 = lop3_and_or(t, kMaskLo, kMagic);
  uint32_t h3 = lop3_and_or(t, kMaskHi, kMagic);
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d[0]) : "r"(h0), "r"(zlo));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d[1]) : "r"(h1), "r"(kSixteenth), "r"(zhi));
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d[2]) : "r"(h2), "r"(zlo));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d[3]) : "r"(h3), "r"(kSixteenth), "r"(zhi));
}

// Rearranges 8 consecutive halves (x = (a0,a1),(a2,a3),(a4,a5),(a6,a7)) into the pairs
// (a0,a4), (a1,a5), (a2,a6), (a3,a7) that line up with nibbles_to_centered_half2.
__device__ __forceinline__ void pair_halves_stride4(const uint4 x, uint32_t p[4]) {
  p[0] = __byte_perm(x.x, x.z, 0x5410);
  p[1] = __byte_perm(x.x, x.z, 0x7632);
  p[2] = __byte_perm(x.y, x.w, 0x5410);
  p[3] = __byte_perm(x.y, x.w, 0x7632);
}

// acc += w.lo * a.lo + w.hi * a.hi with exact fp16 x fp16 products and fp32 sums.
__device__ __forceinline__ float fma2_f16_f32(uint32_t w, uint32_t a, float acc) {
  asm("{\n\t.reg .b16 wl, wh, al, ah;\n\t"
      "mov.b32 {wl, wh}, %1;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "fma.rn.f32.f16 %0, wl, al, %0;\n\t"
      "fma.rn.f32.f16 %0, wh, ah, %0;\n\t}"
      : "+f"(acc)
      : "r"(w), "r"(a));
  return acc;
}

// Output rounding with the optional bias epilogue (matmul_nbits.rs, fold_bias_f16):
// mode 0: fp16(acc); 1: fp16(acc + b) (bias added in fp32, one rounding);
// 2: fp16(fp16(acc) + b) (the accumulator rounded first, as a separate add would).
__device__ __forceinline__ __half round_out(float acc, const __half* bias, int n, int mode) {
  if (mode == 0) return __float2half_rn(acc);
  const float b = __half2float(bias[n]);
  if (mode == 1) return __float2half_rn(acc + b);
  return __float2half_rn(__half2float(__float2half_rn(acc)) + b);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}

// Sum of V per-lane values across a warp, V a power of two <= 32.  Each exchange step
// halves the number of live values per lane, so V values cost V - 1 + (5 - log2 V)
// shuffles.  Afterwards lane L holds the total of value (L >> (5 - log2 V)).
template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[V], int lane) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V must be a power of two");
  int offset = 16;
#pragma unroll
  for (int cnt = V; cnt > 1; cnt >>= 1) {
    const bool upper = (lane & offset) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float keep = upper ? v[i + cnt / 2] : v[i];
      const float send = upper ? v[i] : v[i + cnt / 2];
      v[i] = keep + __shfl_xor_sync(kFull, send, offset);
    }
    offset >>= 1;
  }
  float r = v[0];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (o <= offset) r += __shfl_xor_sync(kFull, r, o);
  }
  return r;
}

}  // namespace mnb

namespace mnb {

// ---------------------------------------------------------------------------------
// mbarrier and 1-D bulk-copy (TMA) helpers.  Every wait is bounded: after
// kSpinLimit polls it gives up and reports failure, so no kernel can hang the GPU
// on a barrier that never completes.
// ---------------------------------------------------------------------------------
constexpr uint32_t kSpinLimit = 1u << 26;

// Device status word codes (OR-ed into the status word by the kernel that gave up).
constexpr uint32_t kStatusFullWait = 1u;   // consumer gave up waiting for a stage
constexpr uint32_t kStatusEmptyWait = 2u;  // producer gave up waiting for a free slot
constexpr uint32_t kStatusMmaWait = 4u;    // tensor-core pipeline wait gave up
constexpr uint32_t kStatusBadIndex = 8u;   // an index input (g_idx, perm, block_group) was out of range

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase with the given parity to complete; false if it gave up (after
// kWaitLimitNs of wall time or kSpinLimit polls, whichever comes first).
constexpr uint64_t kWaitLimitNs = 500ull * 1000 * 1000;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

// As mbar_wait_bounded with a caller-chosen time limit (the poll limit still applies).
__device__ __forceinline__ bool mbar_wait_bounded_ns(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// Spin (no suspension) on the phase: for latency-critical single threads such as the
// MMA issuer.  Bounded like mbar_wait_bounded.
__device__ __forceinline__ bool mbar_spin_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 1023u) == 1023u && global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return false;
}

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned),
// completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Requests the 128-byte line holding p into L1 (a hint: no result, no fault on the line).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

__device__ __forceinline__ void report_status(uint32_t* status, uint32_t code) {
  if (status) atomicOr(status, code);
}

}  // namespace mnb

namespace mnb {

// Shared-memory loads by 32-bit shared-window address.
__device__ __forceinline__ uint4 lds128_a(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8_a(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16_a(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32_a(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_u64_a(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

}  // namespace mnb
