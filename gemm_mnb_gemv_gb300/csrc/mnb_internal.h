// Host-side declarations shared by the mnb translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mnb {

struct QWeight {
  const uint8_t* packed;
  const void* scales;
  const uint8_t* zp;
  int scales_f16;  // 1: fp16 scales, 0: fp32
};

struct LaunchCtx {
  cudaStream_t stream;
  bool pdl;         // launch with programmatic stream serialisation
  int num_sms;
  uint32_t* status = nullptr;     // device status word for bounded waits
  const void* bias = nullptr;     // fp16 [N] or null
  int bias_mode = 0;              // 0 none, 1 fp16(acc + b), 2 fp16(fp16(acc) + b)
  const char* variant = nullptr;  // set by the launcher that ran
};

// Each launcher returns cudaSuccess or the launch error.  Shapes are validated by the
// caller (api.cu).
cudaError_t launch_dequant(LaunchCtx& ctx, const QWeight& w, int K, int N, int bs, float* out);
cudaError_t launch_repack(LaunchCtx& ctx, const uint8_t* packed, int K, int N, uint8_t* out);
// Act-order (g_idx): per-k-group dequant, one-time preparation, per-call activation gather.
cudaError_t launch_dequant_gidx(LaunchCtx& ctx, const QWeight& w, const int32_t* gidx, int K, int N, int bs,
                                float* out);
cudaError_t launch_act_order_prepare(LaunchCtx& ctx, const QWeight& w, int K, int N, int bs, const int32_t* perm,
                                     const int32_t* bgroup, int Kp, uint8_t* packed_out, void* scales_out,
                                     uint8_t* zp_out);
cudaError_t launch_act_order_gather(LaunchCtx& ctx, const void* A, int M, int K, const int32_t* perm, int Kp,
                                    void* out);
// M = 1 act-order GEMV with the gather fused into the activation load (one chunk per lane:
// K' <= 8192); cudaErrorNotSupported otherwise.
cudaError_t launch_gemv_tma_gather(LaunchCtx& ctx, const void* A, const int32_t* perm, int Ka, const QWeight& w,
                                   int Kp, int N, int bs, void* Y);
// The driver's cuTensorMapEncodeTiled (CUDA 12 ABI), or null when unavailable.
void* tensor_map_encode_fn();
// Bulk-copy ring GEMV (M = 1); cudaErrorNotSupported when rows are not 16-byte multiples.
cudaError_t launch_gemv_tma(LaunchCtx& ctx, const void* A, const QWeight& w, int K, int N, int bs,
                            void* Y);
cudaError_t launch_gemv_pair_swiglu_tma(LaunchCtx& ctx, const void* A, const QWeight& gate,
                                        const QWeight& up, int K, int N, int bs, void* out);
// M = 1 GEMV with the multiply-accumulate on mma.sync tensor cores (K % 256 == 0, block
// size 32/64/128); cudaErrorNotSupported for other shapes.
cudaError_t launch_gemv_mma(LaunchCtx& ctx, const void* A, const QWeight& w, int K, int N, int bs, void* Y);
cudaError_t launch_gemv_pair_swiglu_mma(LaunchCtx& ctx, const void* A, const QWeight& gate, const QWeight& up,
                                        int K, int N, int bs, void* out);
// 2 <= M <= 2 * (bs / 32) (block sizes 32 and 64, K % 256 == 0, M * K * 2 <= 32 KB) on the
// M = 1 kernel's machinery with the row mapping; cudaErrorNotSupported otherwise.
cudaError_t launch_gemm_rows_mma(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N, int bs,
                                 void* Y);
// One-thread kernel whose bounded wait on a never-armed mbarrier gives up after limit_ns.
cudaError_t launch_wait_selftest(LaunchCtx& ctx, uint64_t limit_ns);
// Register-pipelined M = 1 GEMV; cudaErrorNotSupported when the shape has no variant.
cudaError_t launch_gemv(LaunchCtx& ctx, const void* A, const QWeight& w, int K, int N, int bs,
                        void* Y);
cudaError_t launch_gemv_pair_swiglu(LaunchCtx& ctx, const void* A, const QWeight& gate,
                                    const QWeight& up, int K, int N, int bs, void* out);
// 2 <= M <= 16 (block size >= 32): weights streamed once, mma.sync over M rows.  For K
// beyond one shared-memory pass the K range is split into slices whose fp32 partials go to
// `workspace` (smallm_workspace_bytes of it) and are summed in slice order.
cudaError_t launch_gemm_smallm(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N, int bs,
                               void* Y, void* workspace, size_t ws_bytes);
int smallm_kslice(int M, int K, int bs, int ssz, bool zp);
size_t smallm_workspace_bytes(int M, int K, int N, int bs);
// M > 16 on the tcgen05 tensor cores, reading the repacked operand.  With a workspace of
// at least gemm_tc_workspace_bytes (the sizing for up to 160 SMs), shapes with fewer
// output tiles than half the SMs split K into slices of whole quant groups and sum their
// fp32 partials in slice order; without one they run unsplit.
cudaError_t launch_gemm_tc(LaunchCtx& ctx, const void* A, int M, const QWeight& w,
                           const uint8_t* repacked, int K, int N, int bs, void* Y, void* workspace = nullptr,
                           size_t ws_bytes = 0);
size_t gemm_tc_workspace_bytes(int M_rows, int K, int N, int bs);
// fp32 activations.  M = 1: bulk-copy GEMV with fp32 activations (K <= 16384).  M >= 2:
// rows split into fp16 hi/lo pairs (A2 holds 2M rows, rexp M exponents), then the small-M
// kernel (2M <= 16) or the tcgen05 kernel with the pair-summing fp32 epilogue.  The generic
// fp32 kernel takes any shape.
cudaError_t launch_gemv_f32_tma(LaunchCtx& ctx, const float* A, const QWeight& w, int K, int N, int bs,
                                float* Y, const float* bias);
cudaError_t launch_split_f32(LaunchCtx& ctx, const float* A, int M, int K, void* A2, int* rexp);
// Fixed-order sums of K-slice partials part[slice][rows][N]: fp16 Y with ctx's bias mode,
// or fp32 Yf from hi/lo row pairs with their exponents (split fp32 activations).
cudaError_t launch_combine_slices(LaunchCtx& ctx, const float* part, int nslices, int M, int N, void* Y);
cudaError_t launch_combine_slices_f32(LaunchCtx& ctx, const float* part, int nslices, int Mout, int N, float* Yf,
                                      const float* biasf, const int* rexp);
cudaError_t launch_gemm_smallm_f32split(LaunchCtx& ctx, const void* A2, int M, const QWeight& w, int K, int N,
                                        int bs, float* Y, const float* bias, const int* rexp,
                                        void* workspace = nullptr, size_t ws_bytes = 0);
cudaError_t launch_gemm_tc_f32split(LaunchCtx& ctx, const void* A2, int M, const QWeight& w,
                                    const uint8_t* repacked, int K, int N, int bs, float* Y, const float* bias,
                                    const int* rexp, void* workspace = nullptr, size_t ws_bytes = 0);
cudaError_t launch_generic_f32(LaunchCtx& ctx, const float* A, int M, const QWeight& w, int K, int N, int bs,
                               float* Y, const float* bias);
// Any M, any K % 16 == 0: CUDA-core kernel, fp32 arithmetic.
cudaError_t launch_generic(LaunchCtx& ctx, const void* A, int M, const QWeight& w, int K, int N,
                           int bs, void* Y);
cudaError_t launch_generic_pair_swiglu(LaunchCtx& ctx, const void* A, const QWeight& gate,
                                       const QWeight& up, int K, int N, int bs, void* out);

// Launch helper: cudaLaunchKernelEx with the programmatic-serialisation attribute when
// ctx.pdl is set.
template <typename Kern, typename... Args>
cudaError_t launch_kernel(LaunchCtx& ctx, Kern kernel, dim3 grid, dim3 block, size_t smem,
                          Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ctx.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace mnb
