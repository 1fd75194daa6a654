// fp64 CPU oracle for block-quantized INT4 (MatMulNBits) products.
//
// TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU baseline
// load this library (through oracle/mnb_oracle.py).  The product library never calls it,
// shares no source, header or table with it, and has no CPU fallback.
//
// What it computes is a plain definition, written out with loops:
//
//     Y[m][n] = sum over k = 0 .. K-1 of  A[m][k] * (code(n, k) - zp(n, g(k))) * scale(n, g(k))
//
// for a weight stored in the ONNX com.microsoft::MatMulNBits layout.  Sources:
//
//   * onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/marlin_gemm.rs, module doc, section
//     "ONNX MatMulNBits int4 format": packed bytes [N][k_blocks][bs/2], the low nibble of a
//     byte holds the even k; scales [N][k_blocks] in fp16 or fp32; zero points packed two
//     per byte, ceil(k_blocks/2) bytes per row, low nibble for the even block; no zero
//     points means 8.
//   * onnx-runtime-ep-cuda 0.1.0-dev.3, src/kernels/matmul_nbits.rs, kernel
//     matmul_nbits_dequant_f32: k_blocks = ceil(K/bs); element (code - zp) * scale written
//     to a [K][N] fp32 matrix at depth * N + n; with act-order group indices the scale and
//     zero point of group g_idx[depth] apply, and a group outside 0 .. k_blocks-1 gives 0.
//
// Arithmetic is fp64.  Codes and zero points are integers in 0..15, fp16 and fp32 scales
// widen exactly, and (code - zp) * scale needs at most 4 + 24 significant bits, so every
// weight is exact; the only rounding in Y is the fp64 sum, taken in ascending k.  With Y
// comes the bound B[m][n] = sum_k |A[m][k] * w[n][k]|: a device result y agrees when
// |y - Y| <= 2e-3 * B + 1e-5.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared -pthread (no fused multiply-add
// contraction, no fast-math; the same results on x86-64 and AArch64).
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------------------
// Storage decoding (marlin_gemm.rs module doc, "ONNX MatMulNBits int4 format")
// ---------------------------------------------------------------------------------------

long long k_blocks(long long K, long long bs) { return (K + bs - 1) / bs; }
long long zp_row_bytes(long long K, long long bs) { return (k_blocks(K, bs) + 1) / 2; }

// The 4-bit code of weight (n, k): byte (n * k_blocks + k / bs) * (bs / 2) + (k % bs) / 2,
// low nibble when k % bs is even, high nibble when it is odd.
int code_at(const uint8_t* packed, long long K, long long bs, long long n, long long k) {
  const long long block = k / bs, within = k % bs;
  const uint8_t byte = packed[(n * k_blocks(K, bs) + block) * (bs / 2) + within / 2];
  return within % 2 == 0 ? (byte & 15) : (byte >> 4);
}

// Zero point of (row n, group g): none stored means 8; else byte n * zp_row_bytes + g / 2,
// low nibble for an even g, high nibble for an odd g.
int zp_at(const uint8_t* zp, long long K, long long bs, long long n, long long g) {
  if (zp == nullptr) return 8;
  const uint8_t byte = zp[n * zp_row_bytes(K, bs) + g / 2];
  return g % 2 == 0 ? (byte & 15) : (byte >> 4);
}

// Exact value of an IEEE-754 binary16 bit pattern: sign s, exponent e, mantissa m;
// e = 0: (-1)^s 2^-14 m/1024; 0 < e < 31: (-1)^s 2^(e-15) (1 + m/1024); e = 31: inf or NaN.
double f16_value(uint16_t h) {
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = std::ldexp((double)m / 1024.0, -14);
  else if (e == 31)
    v = m == 0 ? INFINITY : NAN;
  else
    v = std::ldexp(1.0 + (double)m / 1024.0, e - 15);
  return s ? -v : v;
}

struct Weight {
  const uint8_t* packed;
  const void* scales;
  int scales_f16;        // 1: fp16 scales, 0: fp32 scales
  const uint8_t* zp;     // nullptr: default zero point 8
  const int32_t* g_idx;  // nullptr: group k / bs
  long long K, N, bs;
};

double scale_at(const Weight& w, long long n, long long g) {
  const long long i = n * k_blocks(w.K, w.bs) + g;
  if (w.scales_f16) return f16_value(static_cast<const uint16_t*>(w.scales)[i]);
  return (double)static_cast<const float*>(w.scales)[i];
}

// The group whose scale and zero point apply at k: g_idx[k] with act-order indices
// (matmul_nbits_dequant_f32), else the block k / bs.  The code is always read from block
// k / bs.
long long group_at(const Weight& w, long long k) { return w.g_idx ? (long long)w.g_idx[k] : k / w.bs; }

// w[n][k] = (code - zp) * scale, exact in fp64; 0 for a group outside 0 .. k_blocks-1.
double weight_at(const Weight& w, long long n, long long k) {
  const long long g = group_at(w, k);
  if (g < 0 || g >= k_blocks(w.K, w.bs)) return 0.0;
  const int c = code_at(w.packed, w.K, w.bs, n, k);
  const int z = zp_at(w.zp, w.K, w.bs, n, g);
  return (double)(c - z) * scale_at(w, n, g);
}

// Activation value: fp16 bit patterns decoded exactly, or fp32 widened exactly.
double act_at(const void* A, int a_f16, long long i) {
  if (a_f16) return f16_value(static_cast<const uint16_t*>(A)[i]);
  return (double)static_cast<const float*>(A)[i];
}

// Runs f(i) for i in [0, count) on `threads` threads, each taking a contiguous range.
// Every f(i) writes only its own outputs, so the split changes no result.
template <typename F>
void parallel_for(long long count, int threads, F f) {
  if (threads < 1) threads = 1;
  if (count < (long long)threads) threads = count > 0 ? (int)count : 1;
  if (threads == 1) {
    for (long long i = 0; i < count; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  for (int t = 0; t < threads; ++t) {
    const long long lo = count * t / threads, hi = count * (t + 1) / threads;
    pool.emplace_back([=]() {
      for (long long i = lo; i < hi; ++i) f(i);
    });
  }
  for (auto& th : pool) th.join();
}

// The repacked tensor-core operand (this library's own layout; an independent statement of
// the same specification the device code follows):
//   Np = ceil(N / 128) * 128, Kp = ceil(K / 64) * 64, Np * Kp / 2 bytes.  Row tile t (128
//   rows) and k block b (64 k) own the 4096 bytes at (t * Kp / 64 + b) * 4096.  Inside, the
//   16 bytes at q * 2048 + r * 16 (q = 0, 1; r = 0 .. 127) hold the 32 codes of row
//   n = 128 t + r for k = 64 b + 32 q + i, i = 0 .. 31, as four little-endian 32-bit words:
//   word j = i / 8 holds code i at nibble p (bits 4p .. 4p + 3), where
//   i = 8 j + 2 (p % 4) + p / 4.  Codes of rows n >= N or k >= K are 0.
const long long kRepackRows = 128, kRepackK = 64;

long long repacked_size(long long K, long long N) {
  const long long np = (N + kRepackRows - 1) / kRepackRows * kRepackRows;
  const long long kp = (K + kRepackK - 1) / kRepackK * kRepackK;
  return np * kp / 2;
}

// Byte offset and nibble (0 low, 1 high) of code (n, k) in the repacked buffer.
void repack_position(long long K, long long n, long long k, long long* byte, int* half) {
  const long long kp = (K + kRepackK - 1) / kRepackK * kRepackK;
  const long long t = n / kRepackRows, r = n % kRepackRows;
  const long long b = k / kRepackK, q = (k % kRepackK) / 32, i = k % 32;
  const long long j = i / 8, i8 = i % 8;
  // invert i8 = 2 (p % 4) + p / 4: even i8 -> p = i8 / 2, odd i8 -> p = 4 + i8 / 2
  const long long p = i8 / 2 + 4 * (i8 % 2);
  *byte = (t * (kp / kRepackK) + b) * 4096 + q * 2048 + r * 16 + 4 * j + p / 2;
  *half = (int)(p % 2);
}

}  // namespace

extern "C" {

long long orc_k_blocks(long long K, long long bs) { return k_blocks(K, bs); }
long long orc_zp_row_bytes(long long K, long long bs) { return zp_row_bytes(K, bs); }

// int8 [N][K] codes.
void orc_codes(const uint8_t* packed, long long K, long long N, long long bs, int8_t* out) {
  for (long long n = 0; n < N; ++n)
    for (long long k = 0; k < K; ++k) out[n * K + k] = (int8_t)code_at(packed, K, bs, n, k);
}

// int8 [N][k_blocks] zero points (8 everywhere when zp is null).
void orc_zero_points(const uint8_t* zp, long long K, long long N, long long bs, int8_t* out) {
  const long long G = k_blocks(K, bs);
  for (long long n = 0; n < N; ++n)
    for (long long g = 0; g < G; ++g) out[n * G + g] = (int8_t)zp_at(zp, K, bs, n, g);
}

void orc_f16_to_f64(const uint16_t* h, long long count, double* out) {
  for (long long i = 0; i < count; ++i) out[i] = f16_value(h[i]);
}

// fp64 [N][K] weights w[n][k].
void orc_weight_nk(const uint8_t* packed, const void* scales, int scales_f16, const uint8_t* zp,
                   const int32_t* g_idx, long long K, long long N, long long bs, double* out, int threads) {
  const Weight w{packed, scales, scales_f16, zp, g_idx, K, N, bs};
  parallel_for(N, threads, [&](long long n) {
    for (long long k = 0; k < K; ++k) out[n * K + k] = weight_at(w, n, k);
  });
}

// fp32 [K][N] dequantised weights at depth * N + n (matmul_nbits_dequant_f32): the exact
// fp64 product rounded once to fp32 (exact for fp16 scales; the correctly rounded product
// for fp32 scales).
void orc_dequant_kn_f32(const uint8_t* packed, const void* scales, int scales_f16, const uint8_t* zp,
                        const int32_t* g_idx, long long K, long long N, long long bs, float* out, int threads) {
  const Weight w{packed, scales, scales_f16, zp, g_idx, K, N, bs};
  parallel_for(N, threads, [&](long long n) {
    for (long long k = 0; k < K; ++k) out[k * N + n] = (float)weight_at(w, n, k);
  });
}

// Y[m][n] = sum_k A[m][k] w[n][k] and B[m][n] = sum_k |A[m][k] w[n][k]|, [M][N] fp64, summed
// in ascending k.  A is [M][K], fp16 bit patterns (a_f16 = 1) or fp32.  The output columns
// are split over `threads` threads; each decodes its column's weights once.
void orc_matmul(const void* A, int a_f16, long long M, const uint8_t* packed, const void* scales, int scales_f16,
                const uint8_t* zp, const int32_t* g_idx, long long K, long long N, long long bs, double* Y, double* B,
                int threads) {
  const Weight w{packed, scales, scales_f16, zp, g_idx, K, N, bs};
  std::vector<double> a((size_t)(M * K));
  parallel_for(M, threads, [&](long long m) {
    for (long long k = 0; k < K; ++k) a[(size_t)(m * K + k)] = act_at(A, a_f16, m * K + k);
  });
  parallel_for(N, threads, [&](long long n) {
    std::vector<double> col((size_t)K);
    for (long long k = 0; k < K; ++k) col[(size_t)k] = weight_at(w, n, k);
    for (long long m = 0; m < M; ++m) {
      const double* am = a.data() + m * K;
      double y = 0.0, b = 0.0;
      for (long long k = 0; k < K; ++k) {
        const double prod = am[k] * col[(size_t)k];
        y += prod;
        b += std::fabs(prod);
      }
      Y[m * N + n] = y;
      B[m * N + n] = b;
    }
  });
}

// Y and B as orc_matmul, at the listed (rows[i], cols[i]) pairs only.
void orc_matmul_pairs(const void* A, int a_f16, const uint8_t* packed, const void* scales, int scales_f16,
                      const uint8_t* zp, const int32_t* g_idx, long long K, long long N, long long bs,
                      const long long* rows, const long long* cols, long long count, double* Y, double* B,
                      int threads) {
  const Weight w{packed, scales, scales_f16, zp, g_idx, K, N, bs};
  parallel_for(count, threads, [&](long long i) {
    const long long m = rows[i], n = cols[i];
    double y = 0.0, b = 0.0;
    for (long long k = 0; k < K; ++k) {
      const double prod = act_at(A, a_f16, m * K + k) * weight_at(w, n, k);
      y += prod;
      b += std::fabs(prod);
    }
    Y[i] = y;
    B[i] = b;
  });
}

// silu(x) = x / (1 + exp(-x)), the SwiGLU gate (matmul_nbits.rs,
// matmul_nbits_gemv_f16_gate_up_swiglu).
void orc_silu(const double* x, long long count, double* out) {
  for (long long i = 0; i < count; ++i) out[i] = x[i] / (1.0 + std::exp(-x[i]));
}

// out[i] = silu(g[i]) * u[i].
void orc_swiglu(const double* g, const double* u, long long count, double* out) {
  for (long long i = 0; i < count; ++i) out[i] = g[i] / (1.0 + std::exp(-g[i])) * u[i];
}

long long orc_repacked_bytes(long long K, long long N) { return repacked_size(K, N); }

// Writes the repacked buffer (orc_repacked_bytes bytes, padding nibbles 0).
void orc_repack(const uint8_t* packed, long long K, long long N, long long bs, uint8_t* out) {
  std::memset(out, 0, (size_t)repacked_size(K, N));
  for (long long n = 0; n < N; ++n)
    for (long long k = 0; k < K; ++k) {
      long long byte;
      int half;
      repack_position(K, n, k, &byte, &half);
      out[byte] |= (uint8_t)(code_at(packed, K, bs, n, k) << (4 * half));
    }
}

// int8 [N][K] codes read back from a repacked buffer.
void orc_unrepack_codes(const uint8_t* repacked, long long K, long long N, int8_t* out) {
  for (long long n = 0; n < N; ++n)
    for (long long k = 0; k < K; ++k) {
      long long byte;
      int half;
      repack_position(K, n, k, &byte, &half);
      out[n * K + k] = (int8_t)((repacked[byte] >> (4 * half)) & 15);
    }
}

// Act-order preparation plan (this library's own reading of g_idx; the pages dequantise with
// per-k groups).  Groups in ascending order; inside a group its members in ascending k; each
// group's run padded with empty slots (-1) to whole blocks of bs.  perm[k'] is the source k
// of prepared position k' (or -1), block_group[j] the group of prepared block j.  perm must
// hold K + k_blocks * (bs - 1) entries and block_group that / bs.  Returns K' (the length of
// perm), or -1 with *bad set to the first k whose group is outside 0 .. k_blocks-1 (the
// operator's own check on g_idx in matmul_nbits.rs).
long long orc_act_order_plan(const int32_t* g_idx, long long K, long long bs, int32_t* perm, int32_t* block_group,
                             long long* bad) {
  const long long G = k_blocks(K, bs);
  for (long long k = 0; k < K; ++k)
    if (g_idx[k] < 0 || g_idx[k] >= G) {
      *bad = k;
      return -1;
    }
  long long kp = 0, nb = 0;
  for (long long grp = 0; grp < G; ++grp) {
    long long members = 0;
    for (long long k = 0; k < K; ++k)
      if (g_idx[k] == grp) {
        perm[kp++] = (int32_t)k;
        ++members;
      }
    const long long blocks = (members + bs - 1) / bs;
    for (long long i = members; i < blocks * bs; ++i) perm[kp++] = -1;
    for (long long j = 0; j < blocks; ++j) block_group[nb++] = (int32_t)grp;
  }
  return kp;
}

// The prepared K' x N block weight: codes code(n, perm[k']) (the block's zero point at an
// empty slot, so that weight is 0), packed two per byte with the even k' low; scales of
// block j copied from group block_group[j] (scale_bytes 2 or 4 per value); zero points of
// block j those of block_group[j], packed two per byte (the unused high nibble of an odd
// block count is 0), written only when zp is not null.
void orc_act_order_prepare(const uint8_t* packed, const void* scales, int scale_bytes, const uint8_t* zp, long long K,
                           long long N, long long bs, const int32_t* perm, const int32_t* block_group, long long Kp,
                           uint8_t* packed_out, void* scales_out, uint8_t* zp_out) {
  const long long G = k_blocks(K, bs), Gp = Kp / bs, zrbp = (Gp + 1) / 2;
  for (long long n = 0; n < N; ++n) {
    for (long long kk = 0; kk < Kp; kk += 2) {
      int c[2];
      for (int h = 0; h < 2; ++h) {
        const long long k2 = kk + h;
        const long long grp = block_group[k2 / bs];
        c[h] = perm[k2] >= 0 ? code_at(packed, K, bs, n, perm[k2]) : zp_at(zp, K, bs, n, grp);
      }
      packed_out[n * (Kp / 2) + kk / 2] = (uint8_t)(c[0] | (c[1] << 4));
    }
    for (long long j = 0; j < Gp; ++j)
      std::memcpy(static_cast<uint8_t*>(scales_out) + (n * Gp + j) * scale_bytes,
                  static_cast<const uint8_t*>(scales) + (n * G + block_group[j]) * scale_bytes, (size_t)scale_bytes);
    if (zp != nullptr && zp_out != nullptr) {
      for (long long jb = 0; jb < zrbp; ++jb) {
        const int lo = zp_at(zp, K, bs, n, block_group[2 * jb]);
        const int hi = 2 * jb + 1 < Gp ? zp_at(zp, K, bs, n, block_group[2 * jb + 1]) : 0;
        zp_out[n * zrbp + jb] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

// A'[m][k'] = A[m][perm[k']], and all-zero bits (+0) where perm[k'] = -1; elements of
// elem_bytes bytes (2 for fp16, 4 for fp32).
void orc_act_order_gather(const void* A, long long M, long long K, int elem_bytes, const int32_t* perm, long long Kp,
                          void* out) {
  const uint8_t* src = static_cast<const uint8_t*>(A);
  uint8_t* dst = static_cast<uint8_t*>(out);
  for (long long m = 0; m < M; ++m)
    for (long long kk = 0; kk < Kp; ++kk) {
      uint8_t* d = dst + (m * Kp + kk) * elem_bytes;
      if (perm[kk] >= 0)
        std::memcpy(d, src + (m * K + perm[kk]) * elem_bytes, (size_t)elem_bytes);
      else
        std::memset(d, 0, (size_t)elem_bytes);
    }
}

}  // extern "C"
