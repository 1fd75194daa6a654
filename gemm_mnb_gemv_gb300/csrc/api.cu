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

// M = 1: the bulk-copy ring kernel when rows are 16-byte multiples, else the
// register-pipelined kernel, else the generic kernel.
cudaError_t run_gemv(mnb::LaunchCtx& ctx, const void* A, const mnb::QWeight& q, int K, int N, int bs,
                     void* Y) {
  cudaError_t e = mnb::launch_gemv_tma(ctx, A, q, K, N, bs, Y);
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
  return fail(MNB_ERR_TIMEOUT, "%s: a device-side wait gave up (status bits 0x%x: 1 = stage wait, "
              "2 = slot wait, 4 = tensor-core pipeline wait); outputs of that call are NaN", fn, v);
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
  (void)M;
  (void)K;
  (void)N;
  (void)block_size;
  return 0;
}

}  // extern "C"

namespace {

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
  const size_t need = mnb_workspace_bytes(M, K, N, block_size);
  if (ws_bytes < need)
    return fail(MNB_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", fn, ws_bytes, need);
  if (need > 0 && (st = check_ptr(fn, "workspace", workspace)) != MNB_OK) return st;
  if (M > 16) {
    if ((st = check_ptr(fn, "repacked", repacked)) != MNB_OK) return st;
  }
  if (bias_mode < 0 || bias_mode > 2)
    return fail(MNB_ERR_INVALID_ARG, "%s: bias_mode %d must be 0, 1 or 2", fn, bias_mode);
  if (bias_mode != 0 && (st = check_ptr(fn, "bias", bias)) != MNB_OK) return st;
  mnb::LaunchCtx ctx;
  if ((st = make_ctx(fn, stream, &ctx)) != MNB_OK) return st;
  ctx.bias = bias_mode ? bias : nullptr;
  ctx.bias_mode = bias_mode;
  cudaError_t e;
  if (M == 1) {
    e = run_gemv(ctx, A, q, K, N, block_size, Y);
  } else if (M > 16) {
    e = mnb::launch_gemm_tc(ctx, A, M, q, repacked, K, N, block_size, Y);
    if (e == cudaErrorNotSupported) e = mnb::launch_generic(ctx, A, M, q, K, N, block_size, Y);
  } else {
    e = mnb::launch_gemm_smallm(ctx, A, M, q, K, N, block_size, Y);
    if (e == cudaErrorNotSupported) e = mnb::launch_generic(ctx, A, M, q, K, N, block_size, Y);
  }
  return finish(fn, e, ctx);
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
  cudaError_t e = mnb::launch_gemv_pair_swiglu_tma(ctx, A, g, u, K, N, block_size, out);
  if (e == cudaErrorNotSupported) e = mnb::launch_gemv_pair_swiglu(ctx, A, g, u, K, N, block_size, out);
  if (e == cudaErrorNotSupported) e = mnb::launch_generic_pair_swiglu(ctx, A, g, u, K, N, block_size, out);
  return finish(fn, e, ctx);
}

}  // extern "C"
