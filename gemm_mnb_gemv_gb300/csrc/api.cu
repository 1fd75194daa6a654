// C ABI of libmnb: argument validation, error reporting and kernel dispatch.
//
// Validation follows the attribute and shape rules of the MatMulNBits operator
// (matmul_nbits.rs, MatMulNBitsFactory::create: bits = 4, block_size a power of two
// >= 16; marlin_gemm.rs, launch_marlin_gemm: K a multiple of 16 and of the group size,
// sizes that fit 32-bit indices), with every failure returned as a status code and a
// message instead of an exception (the EpError::KernelFailed strings of matmul_nbits.rs).
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "mnb.h"
#include "mnb_internal.h"

namespace {

thread_local std::string g_last_error;

// Set (bitwise OR) by a kernel whose bounded device-side wait gave up.
__device__ uint32_t g_device_status;
std::mutex g_status_mu;
uint32_t* g_status_ptr[128] = {};

uint32_t* device_status_ptr(int dev) {
  if (dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_status_ptr[dev];
}
thread_local const char* g_last_variant = "";
thread_local bool g_pdl = false;

mnb_status fail(mnb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mnb_status cuda_fail(const char* what, cudaError_t e) {
  return fail(MNB_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxKN = 1 << 24;
constexpr int kMaxM = 1 << 20;

mnb_status check_shape(const char* fn, int K, int N, int bs) {
  if (!(bs == 16 || bs == 32 || bs == 64 || bs == 128))
    return fail(MNB_ERR_INVALID_ARG, "%s: block_size %d must be 16, 32, 64 or 128", fn, bs);
  if (K < 1 || N < 1 || K > kMaxKN || N > kMaxKN)
    return fail(MNB_ERR_INVALID_ARG, "%s: K=%d and N=%d must be in [1, 2^24]", fn, K, N);
  if (K % bs != 0)
    return fail(MNB_ERR_UNSUPPORTED, "%s: K=%d is not a multiple of block_size %d", fn, K, bs);
  return MNB_OK;
}

mnb_status check_ptr(const char* fn, const char* name, const void* p) {
  if (!p) return fail(MNB_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
  if (!aligned16(p)) return fail(MNB_ERR_MISALIGNED, "%s: %s is not 16-byte aligned", fn, name);
  return MNB_OK;
}

mnb_status check_weight(const char* fn, const mnb_weight& w, mnb::QWeight* q) {
  mnb_status st;
  if ((st = check_ptr(fn, "packed", w.packed)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "scales", w.scales)) != MNB_OK) return st;
  if (w.zero_points && !aligned16(w.zero_points))
    return fail(MNB_ERR_MISALIGNED, "%s: zero_points is not 16-byte aligned", fn);
  if (w.scales_dtype != MNB_F16 && w.scales_dtype != MNB_F32)
    return fail(MNB_ERR_INVALID_ARG, "%s: scales_dtype %d must be MNB_F16 or MNB_F32", fn,
                (int)w.scales_dtype);
  q->packed = w.packed;
  q->scales = w.scales;
  q->zp = w.zero_points;
  q->scales_f16 = w.scales_dtype == MNB_F16 ? 1 : 0;
  return MNB_OK;
}

mnb_status make_ctx(const char* fn, mnb_stream stream, mnb::LaunchCtx* ctx) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  ctx->stream = reinterpret_cast<cudaStream_t>(stream);
  ctx->pdl = g_pdl;
  ctx->num_sms = sms;
  ctx->status = device_status_ptr(dev);
  ctx->variant = nullptr;
  return MNB_OK;
}

// M = 1: the tensor-core streaming kernel (K % 256 == 0, block size 32/64/128), else the
// bulk-copy ring kernel when rows are 16-byte multiples, else the register-pipelined
// kernel, else the generic kernel.
cudaError_t run_gemv(mnb::LaunchCtx& ctx, const void* A, const mnb::QWeight& q, int K, int N, int bs,
                     void* Y) {
  cudaError_t e = mnb::launch_gemv_mma(ctx, A, q, K, N, bs, Y);
  if (e == cudaErrorNotSupported) e = mnb::launch_gemv_tma(ctx, A, q, K, N, bs, Y);
  if (e == cudaErrorNotSupported) e = mnb::launch_gemv(ctx, A, q, K, N, bs, Y);
  if (e == cudaErrorNotSupported) e = mnb::launch_generic(ctx, A, 1, q, K, N, bs, Y);
  return e;
}

mnb_status finish(const char* fn, cudaError_t e, const mnb::LaunchCtx& ctx) {
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(fn, e);
  g_last_variant = ctx.variant ? ctx.variant : "";
  g_last_error.clear();
  return MNB_OK;
}

}  // namespace

extern "C" {

const char* mnb_last_error(void) { return g_last_error.c_str(); }
const char* mnb_last_variant(void) { return g_last_variant; }
const char* mnb_version(void) { return "mnb 0.1.0 (sm_103a)"; }
void mnb_set_programmatic_launch(int enable) { g_pdl = enable != 0; }

mnb_status mnb_check_device_status(void) {
  const char* fn = "mnb_check_device_status";
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(fn, e);
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (v == 0) {
    g_last_error.clear();
    return MNB_OK;
  }
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (v & 7u)
    return fail(MNB_ERR_TIMEOUT, "%s: a device-side wait gave up (status bits 0x%x: 1 = stage wait, "
                "2 = slot wait, 4 = tensor-core pipeline wait, 8 = index out of range); outputs of that "
                "call are NaN", fn, v);
  return fail(MNB_ERR_INVALID_ARG, "%s: an index input was out of range (status bits 0x%x: a g_idx, perm "
              "or block_group entry outside its range; that element was written as 0)", fn, v);
}

mnb_status mnb_selftest_wait_timeout(unsigned int limit_us, mnb_stream stream) {
  const char* fn = "mnb_selftest_wait_timeout";
  if (limit_us < 1 || limit_us > 1000000)
    return fail(MNB_ERR_INVALID_ARG, "%s: limit_us = %u is outside 1 .. 1000000", fn, limit_us);
  mnb::LaunchCtx ctx;
  mnb_status st;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn, mnb::launch_wait_selftest(ctx, (uint64_t)limit_us * 1000ull), ctx);
}

mnb_status mnb_dequant(mnb_weight w, int K, int N, int block_size, float* out_kn,
                       mnb_stream stream) {
  const char* fn = "mnb_dequant";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "out_kn", out_kn)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn, mnb::launch_dequant(ctx, q, K, N, block_size, out_kn), ctx);
}

size_t mnb_repacked_bytes(int K, int N, int block_size) {
  if (!(block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128)) return 0;
  if (K < 1 || N < 1 || K > kMaxKN || N > kMaxKN || K % block_size != 0) return 0;
  const size_t np = (size_t)((N + 127) / 128) * 128;
  const size_t kp = (size_t)((K + 63) / 64) * 64;
  return np * kp / 2;
}

mnb_status mnb_repack(const uint8_t* packed, int K, int N, int block_size, uint8_t* out,
                      mnb_stream stream) {
  const char* fn = "mnb_repack";
  mnb_status st;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "packed", packed)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "out", out)) != MNB_OK) return st;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (cs != cudaStreamCaptureStatusNone)
    return fail(MNB_ERR_CAPTURE, "%s: refused while the stream is capturing; repack once, "
                "before capture", fn);
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn, mnb::launch_repack(ctx, packed, K, N, out), ctx);
}

mnb_status mnb_gemv(const void* A, mnb_weight w, int K, int N, int block_size, void* Y,
                    mnb_stream stream) {
  const char* fn = "mnb_gemv";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "Y", Y)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn, run_gemv(ctx, A, q, K, N, block_size, Y), ctx);
}

size_t mnb_workspace_bytes(int M, int K, int N, int block_size) {
  // fp32 K-slice partials: required by the small-M kernel when K exceeds one shared-memory
  // pass; for M > 16 the tensor-core kernel uses them, when given, to split K over the SMs
  // for outputs with few tiles.
  if (M < 2 || M > kMaxM || K < 1 || N < 1 || K > kMaxKN || N > kMaxKN) return 0;
  if (M > 16) return mnb::gemm_tc_workspace_bytes(M, K, N, block_size);
  return mnb::smallm_workspace_bytes(M, K, N, block_size);
}

}  // extern "C"

namespace {

// M = 1: GEMV; M > 16: tcgen05 GEMM on the repacked operand; otherwise the row mapping of
// the GEMV kernel or the small-M kernel.  Shapes no specialised kernel takes go to the
// generic kernel.
cudaError_t dispatch_gemm(mnb::LaunchCtx& ctx, const void* A, int M, const mnb::QWeight& q,
                          const uint8_t* repacked, int K, int N, int bs, void* Y, void* workspace = nullptr,
                          size_t ws_bytes = 0) {
  cudaError_t e;
  if (M == 1) {
    e = run_gemv(ctx, A, q, K, N, bs, Y);
  } else if (M > 16) {
    e = mnb::launch_gemm_tc(ctx, A, M, q, repacked, K, N, bs, Y, workspace, ws_bytes);
    if (e == cudaErrorNotSupported) e = mnb::launch_generic(ctx, A, M, q, K, N, bs, Y);
  } else {
    // rows on the M = 1 kernel's machinery where its row mapping takes them (M <= 2 or 4 at
    // block sizes 32 or 64), else the small-M kernel
    e = mnb::launch_gemm_rows_mma(ctx, A, M, q, K, N, bs, Y);
    if (e == cudaErrorNotSupported) e = mnb::launch_gemm_smallm(ctx, A, M, q, K, N, bs, Y, workspace, ws_bytes);
    if (e == cudaErrorNotSupported) e = mnb::launch_generic(ctx, A, M, q, K, N, bs, Y);
  }
  return e;
}

mnb_status check_bias(const char* fn, const void* bias, int bias_mode) {
  if (bias_mode < 0 || bias_mode > 2)
    return fail(MNB_ERR_INVALID_ARG, "%s: bias_mode %d must be 0, 1 or 2", fn, bias_mode);
  if (bias_mode != 0) return check_ptr(fn, "bias", bias);
  return MNB_OK;
}

mnb_status gemm_impl(const char* fn, const void* A, int M, mnb_weight w, const uint8_t* repacked, int K, int N,
                     int block_size, const void* bias, int bias_mode, void* workspace, size_t ws_bytes, void* Y,
                     mnb_stream stream) {
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_INVALID_ARG, "%s: M=%d must be in [1, 2^20]", fn, M);
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "Y", Y)) != MNB_OK) return st;
  // Required for 2 <= M <= 16; optional (a K split when it fits) for M > 16.
  const size_t need = M <= 16 ? mnb_workspace_bytes(M, K, N, block_size) : 0;
  if (ws_bytes < need)
    return fail(MNB_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
  if ((need > 0 || (workspace && ws_bytes > 0)) && (st = check_ptr(fn, "workspace", workspace)) != MNB_OK) return st;
  if (M > 16) {
    if ((st = check_ptr(fn, "repacked", repacked)) != MNB_OK) return st;
  }
  if ((st = check_bias(fn, bias, bias_mode)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  ctx.bias = bias_mode ? bias : nullptr;
  ctx.bias_mode = bias_mode;
  return finish(fn, dispatch_gemm(ctx, A, M, q, repacked, K, N, block_size, Y, workspace, ws_bytes), ctx);
}

}  // namespace

extern "C" {

mnb_status mnb_gemm(const void* A, int M, mnb_weight w, const uint8_t* repacked, int K, int N,
                    int block_size, void* workspace, size_t ws_bytes, void* Y,
                    mnb_stream stream) {
  return gemm_impl("mnb_gemm", A, M, w, repacked, K, N, block_size, nullptr, 0, workspace, ws_bytes, Y,
                   stream);
}

mnb_status mnb_gemm_bias(const void* A, int M, mnb_weight w, const uint8_t* repacked, int K, int N,
                         int block_size, const void* bias, int bias_mode, void* workspace, size_t ws_bytes,
                         void* Y, mnb_stream stream) {
  return gemm_impl("mnb_gemm_bias", A, M, w, repacked, K, N, block_size, bias, bias_mode, workspace,
                   ws_bytes, Y, stream);
}

mnb_status mnb_gemv_gate_up_swiglu(const void* A, mnb_weight gate, mnb_weight up, int K, int N,
                                   int block_size, void* out, mnb_stream stream) {
  const char* fn = "mnb_gemv_gate_up_swiglu";
  mnb_status st;
  mnb::QWeight g, u;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if ((st = check_weight(fn, gate, &g)) != MNB_OK) return st;
  if ((st = check_weight(fn, up, &u)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "out", out)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  cudaError_t e = mnb::launch_gemv_pair_swiglu_mma(ctx, A, g, u, K, N, block_size, out);
  if (e == cudaErrorNotSupported) e = mnb::launch_gemv_pair_swiglu_tma(ctx, A, g, u, K, N, block_size, out);
  if (e == cudaErrorNotSupported) e = mnb::launch_gemv_pair_swiglu(ctx, A, g, u, K, N, block_size, out);
  if (e == cudaErrorNotSupported) e = mnb::launch_generic_pair_swiglu(ctx, A, g, u, K, N, block_size, out);
  return finish(fn, e, ctx);
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// fp32 activations.
// ------------------------------------------------------------------------------------

extern "C" {

size_t mnb_workspace_bytes_f32(int M, int K, int N, int block_size) {
  if (M < 2 || M > kMaxM || K < 1 || K > kMaxKN || N < 1 || N > kMaxKN) return 0;
  const size_t split = (size_t)4 * (size_t)M * (size_t)K;           // 2M fp16 rows of K
  size_t bytes = split + ((size_t)4 * (size_t)M + 15) / 16 * 16;    // + M exponents
  // + K-slice partials of the 2M split rows (required on the small-M kernel, optional on
  // the tensor-core kernel)
  bytes += 2 * M <= 16 ? mnb::smallm_workspace_bytes(2 * M, K, N, block_size)
                       : mnb::gemm_tc_workspace_bytes(2 * M, K, N, block_size);
  return bytes;
}

mnb_status mnb_gemm_f32(const float* A, int M, mnb_weight w, const uint8_t* repacked, int K, int N, int block_size,
                        const float* bias, void* workspace, size_t ws_bytes, float* Y, mnb_stream stream) {
  const char* fn = "mnb_gemm_f32";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_INVALID_ARG, "%s: M=%d must be in [1, 2^20]", fn, M);
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "Y", Y)) != MNB_OK) return st;
  if (bias && !aligned16(bias)) return fail(MNB_ERR_MISALIGNED, "%s: bias is not 16-byte aligned", fn);
  // Required: the split activation and exponents, plus the small-M kernel's partials; the
  // tensor-core kernel's partials (2M > 16) are optional.
  size_t need = mnb_workspace_bytes_f32(M, K, N, block_size);
  if (2 * M > 16) need -= mnb::gemm_tc_workspace_bytes(2 * M, K, N, block_size);
  if (ws_bytes < need)
    return fail(MNB_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
  if (need > 0 && (st = check_ptr(fn, "workspace", workspace)) != MNB_OK) return st;
  if (2 * M > 16 && (st = check_ptr(fn, "repacked", repacked)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  cudaError_t e;
  if (M == 1) {
    e = mnb::launch_gemv_f32_tma(ctx, A, q, K, N, block_size, Y, bias);
  } else {
    uint8_t* a2 = static_cast<uint8_t*>(workspace);
    int* rexp = reinterpret_cast<int*>(a2 + (size_t)4 * M * K);
    const size_t head = (size_t)4 * M * K + ((size_t)4 * M + 15) / 16 * 16;
    e = mnb::launch_split_f32(ctx, A, M, K, a2, rexp);
    if (e == cudaSuccess) {
      if (2 * M <= 16)
        e = mnb::launch_gemm_smallm_f32split(ctx, a2, M, q, K, N, block_size, Y, bias, rexp, a2 + head,
                                             ws_bytes - head);
      else
        e = mnb::launch_gemm_tc_f32split(ctx, a2, M, q, repacked, K, N, block_size, Y, bias, rexp, a2 + head,
                                         ws_bytes - head);
    }
  }
  if (e == cudaErrorNotSupported) e = mnb::launch_generic_f32(ctx, A, M, q, K, N, block_size, Y, bias);
  return finish(fn, e, ctx);
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// Act-order (g_idx) weights.
// ------------------------------------------------------------------------------------

namespace {

mnb_status refuse_capture(const char* fn, mnb_stream stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (cs != cudaStreamCaptureStatusNone)
    return fail(MNB_ERR_CAPTURE, "%s: refused while the stream is capturing; prepare once, before capture", fn);
  return MNB_OK;
}

// K <= K' <= 2K holds for every plan (each non-empty group adds fewer than bs slots,
// and there are at most K / bs groups).
mnb_status check_prepared_k(const char* fn, int K, int Kp, int bs) {
  mnb_status st;
  if ((st = check_shape(fn, Kp, 1, bs)) != MNB_OK) return st;
  if (K < 1 || K > kMaxKN || K % bs != 0)
    return fail(MNB_ERR_INVALID_ARG, "%s: K=%d must be a multiple of block_size %d in [1, 2^24]", fn, K, bs);
  if (Kp < K || Kp > 2 * K)
    return fail(MNB_ERR_INVALID_ARG, "%s: K_prepared=%d must lie in [K, 2K] for K=%d", fn, Kp, K);
  return MNB_OK;
}

}  // namespace

extern "C" {

mnb_status mnb_act_order_plan(const int32_t* g_idx, int K, int block_size, int32_t* K_prepared, int32_t* perm,
                              int32_t* block_group) {
  const char* fn = "mnb_act_order_plan";
  mnb_status st;
  if ((st = check_shape(fn, K, 1, block_size)) != MNB_OK) return st;
  if (!g_idx) return fail(MNB_ERR_INVALID_ARG, "%s: g_idx is NULL", fn);
  if (!K_prepared) return fail(MNB_ERR_INVALID_ARG, "%s: K_prepared is NULL", fn);
  const int G = K / block_size;
  std::vector<int64_t> count(G, 0);
  for (int k = 0; k < K; ++k) {
    const int32_t g = g_idx[k];
    if (g < 0 || g >= G)
      return fail(MNB_ERR_INVALID_ARG, "%s: g_idx[%d]=%d is outside 0..%d", fn, k, (int)g, G);
    ++count[g];
  }
  // Each group's run starts at a block boundary; its slots past the members stay -1.
  std::vector<int64_t> start(G + 1, 0);
  for (int g = 0; g < G; ++g)
    start[g + 1] = start[g] + (count[g] + block_size - 1) / block_size * block_size;
  const int64_t kp = start[G];
  *K_prepared = (int32_t)kp;
  if (perm) {
    std::vector<int64_t> cursor(start.begin(), start.end() - 1);
    for (int64_t i = 0; i < kp; ++i) perm[i] = -1;
    for (int k = 0; k < K; ++k) perm[cursor[g_idx[k]]++] = k;
  }
  if (block_group) {
    for (int g = 0; g < G; ++g)
      for (int64_t j = start[g] / block_size; j < start[g + 1] / block_size; ++j) block_group[j] = g;
  }
  g_last_error.clear();
  return MNB_OK;
}

mnb_status mnb_dequant_gidx(mnb_weight w, const int32_t* g_idx, int K, int N, int block_size, float* out_kn,
                            mnb_stream stream) {
  const char* fn = "mnb_dequant_gidx";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "g_idx", g_idx)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "out_kn", out_kn)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn, mnb::launch_dequant_gidx(ctx, q, g_idx, K, N, block_size, out_kn), ctx);
}

mnb_status mnb_act_order_prepare(mnb_weight w, int K, int N, int block_size, const int32_t* perm,
                                 const int32_t* block_group, int K_prepared, uint8_t* packed_out,
                                 void* scales_out, uint8_t* zero_points_out, mnb_stream stream) {
  const char* fn = "mnb_act_order_prepare";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K, N, block_size)) != MNB_OK) return st;
  if ((st = check_prepared_k(fn, K, K_prepared, block_size)) != MNB_OK) return st;
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "perm", perm)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "block_group", block_group)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "packed_out", packed_out)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "scales_out", scales_out)) != MNB_OK) return st;
  if (w.zero_points && (st = check_ptr(fn, "zero_points_out", zero_points_out)) != MNB_OK) return st;
  if ((st = refuse_capture(fn, stream)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn,
                mnb::launch_act_order_prepare(ctx, q, K, N, block_size, perm, block_group, K_prepared,
                                              packed_out, scales_out, w.zero_points ? zero_points_out : nullptr),
                ctx);
}

mnb_status mnb_act_order_gather(const void* A, int M, int K, const int32_t* perm, int K_prepared, void* A_out,
                                mnb_stream stream) {
  const char* fn = "mnb_act_order_gather";
  mnb_status st;
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_INVALID_ARG, "%s: M=%d must be in [1, 2^20]", fn, M);
  if (K < 1 || K > kMaxKN) return fail(MNB_ERR_INVALID_ARG, "%s: K=%d must be in [1, 2^24]", fn, K);
  if (K_prepared < 8 || K_prepared % 8 != 0 || K_prepared > 2 * K)
    return fail(MNB_ERR_INVALID_ARG, "%s: K_prepared=%d must be a positive multiple of 8, at most 2K", fn,
                K_prepared);
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "perm", perm)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A_out", A_out)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  return finish(fn, mnb::launch_act_order_gather(ctx, A, M, K, perm, K_prepared, A_out), ctx);
}

size_t mnb_act_order_workspace_bytes(int M, int K_prepared) {
  if (M < 1 || M > kMaxM || K_prepared < 1 || K_prepared > 2 * kMaxKN) return 0;
  return (size_t)M * (size_t)K_prepared * 2;
}

mnb_status mnb_gemm_act_order(const void* A, int M, mnb_weight w, const uint8_t* repacked, const int32_t* perm,
                              int K, int K_prepared, int N, int block_size, const void* bias, int bias_mode,
                              void* workspace, size_t ws_bytes, void* Y, mnb_stream stream) {
  const char* fn = "mnb_gemm_act_order";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K_prepared, N, block_size)) != MNB_OK) return st;
  if ((st = check_prepared_k(fn, K, K_prepared, block_size)) != MNB_OK) return st;
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_INVALID_ARG, "%s: M=%d must be in [1, 2^20]", fn, M);
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "perm", perm)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "Y", Y)) != MNB_OK) return st;
  if (M > 16 && (st = check_ptr(fn, "repacked", repacked)) != MNB_OK) return st;
  if ((st = check_bias(fn, bias, bias_mode)) != MNB_OK) return st;
  const size_t need = mnb_act_order_workspace_bytes(M, K_prepared);
  if (ws_bytes < need)
    return fail(MNB_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
  if ((st = check_ptr(fn, "workspace", workspace)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  ctx.bias = bias_mode ? bias : nullptr;
  ctx.bias_mode = bias_mode;
  // M = 1: the GEMV gathers its activations itself (no second launch, workspace unused).
  cudaError_t e = M == 1 ? mnb::launch_gemv_tma_gather(ctx, A, perm, K, q, K_prepared, N, block_size, Y)
                         : cudaErrorNotSupported;
  if (e == cudaErrorNotSupported) {
    e = mnb::launch_act_order_gather(ctx, A, M, K, perm, K_prepared, workspace);
    // Workspace beyond the gathered activation (rounded to 16 bytes) serves the small-M
    // kernel's K-slice partials when K' exceeds one shared-memory pass.
    const size_t head = (need + 15) / 16 * 16;
    void* rest = ws_bytes > head ? static_cast<uint8_t*>(workspace) + head : nullptr;
    if (e == cudaSuccess)
      e = dispatch_gemm(ctx, workspace, M, q, repacked, K_prepared, N, block_size, Y, rest,
                        rest ? ws_bytes - head : 0);
  }
  return finish(fn, e, ctx);
}

}  // extern "C"

// ------------------------------------------------------------------------------------
// Act-order product for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin inside a host framework that owns all
// device memory through its own allocator and hands the plugin no workspace, or a
// latency-critical loop where cudaMalloc's implicit device synchronisation is not
// allowed. mnb_gemm_act_order_noalloc takes its scratch (the gathered activation
// A'[M, K'] in fp16) from the fixed array below instead of a caller workspace.
// ------------------------------------------------------------------------------------

// 8 MiB: M * K' * 2 bytes must fit (e.g. M = 16 with K' up to 262144, M = 1024 with
// K' = 4096). Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[128] = {};

// Once per device, with that device current: the device address of g_noalloc_scratch
// (in host code the array's name is only a stand-in for the symbol, not an address).
mnb_status noalloc_scratch(const char* fn, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(fn, e);
  if (dev < 0 || dev >= 128) return fail(MNB_ERR_UNSUPPORTED, "%s: device ordinal %d is above 127", fn, dev);
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(fn, e);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MNB_OK;
}

}  // namespace

extern "C" {

mnb_status mnb_gemm_act_order_noalloc(const void* A, int M, mnb_weight w, const uint8_t* repacked,
                                      const int32_t* perm, int K, int K_prepared, int N, int block_size,
                                      const void* bias, int bias_mode, void* Y, mnb_stream stream) {
  const char* fn = "mnb_gemm_act_order_noalloc";
  mnb_status st;
  mnb::QWeight q;
  if ((st = check_shape(fn, K_prepared, N, block_size)) != MNB_OK) return st;
  if ((st = check_prepared_k(fn, K, K_prepared, block_size)) != MNB_OK) return st;
  if (M < 1 || M > kMaxM) return fail(MNB_ERR_INVALID_ARG, "%s: M=%d must be in [1, 2^20]", fn, M);
  if ((st = check_weight(fn, w, &q)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "A", A)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "perm", perm)) != MNB_OK) return st;
  if ((st = check_ptr(fn, "Y", Y)) != MNB_OK) return st;
  if (M > 16 && (st = check_ptr(fn, "repacked", repacked)) != MNB_OK) return st;
  if ((st = check_bias(fn, bias, bias_mode)) != MNB_OK) return st;
  const size_t need = (size_t)M * (size_t)K_prepared * 2;
  if (need > kNoAllocScratchBytes)
    return fail(MNB_ERR_UNSUPPORTED, "%s: M=%d x K_prepared=%d needs %zu scratch bytes; the library's static "
                "scratch holds %zu (use mnb_gemm_act_order with a workspace)", fn, M, K_prepared, need,
                kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = noalloc_scratch(fn, &scratch)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  // When the gather pass runs (M > 1, or K' beyond the fused GEMV) it writes every byte
  // of A'[M, K'] that the product then reads, padding slots included, so nothing left in
  // the array by an earlier call is used.
  ctx.bias = bias_mode ? bias : nullptr;
  ctx.bias_mode = bias_mode;
  cudaError_t e = M == 1 ? mnb::launch_gemv_tma_gather(ctx, A, perm, K, q, K_prepared, N, block_size, Y)
                         : cudaErrorNotSupported;
  if (e == cudaErrorNotSupported) {
    e = mnb::launch_act_order_gather(ctx, A, M, K, perm, K_prepared, scratch);
    // The rest of the scratch serves the small-M kernel's K-slice partials.
    const size_t head = (need + 15) / 16 * 16;
    if (e == cudaSuccess)
      e = dispatch_gemm(ctx, scratch, M, q, repacked, K_prepared, N, block_size, Y,
                        static_cast<uint8_t*>(scratch) + head, kNoAllocScratchBytes - head);
  }
  return finish(fn, e, ctx);
}

}  // extern "C"
