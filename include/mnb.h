/*
 * mnb.h -- block-quantized INT4 (MatMulNBits) products on one GB300 GPU (sm_103a).
 *
 * The library computes Y[M,N] = A[M,K] . dequant(B)^T for weights stored in the
 * ONNX com.microsoft::MatMulNBits layout, as spelled out in
 *   onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/marlin_gemm.rs, module doc,
 *   section "ONNX MatMulNBits int4 format", and
 *   onnx-runtime-ep-cuda 0.1.0-dev.3, src/kernels/matmul_nbits.rs, kernel
 *   matmul_nbits_dequant_f32:
 *
 *   packed       uint8 [N, k_blocks, bs/2], k_blocks = K/bs. The nibble for (n, k) is in
 *                byte (n*k_blocks + k/bs)*(bs/2) + (k%bs)/2: low nibble for even k,
 *                high nibble for odd k. code in 0..15. (With K % bs == 0 every row is
 *                simply K/2 consecutive bytes.)
 *   scales       [N, k_blocks], fp16 or fp32.
 *   zero_points  optional uint8 [N, ceil(k_blocks/2)]: the nibble for (n, g) is in byte
 *                n*ceil(k_blocks/2) + g/2, low nibble for even g. NULL means zp = 8.
 *   dequant(B)[n, k] = (code[n, k] - zp[n, k/bs]) * scale[n, k/bs].
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is device memory owned by the caller (except where an
 *     argument is marked HOST); the library keeps no reference after the call returns
 *     and allocates nothing.
 *   - A and Y are fp16 (IEEE binary16, passed as raw 16-bit storage), row-major, except
 *     in mnb_gemm_f32, where they are fp32.
 *   - Every device pointer must be non-NULL (except zero_points, workspace when
 *     ws_bytes is 0, and repacked where stated) and 16-byte aligned:
 *     otherwise MNB_ERR_INVALID_ARG / MNB_ERR_MISALIGNED.
 *   - block_size must be 16, 32, 64 or 128 and K a multiple of it; K, N, M >= 1 and
 *     K, N <= 2^24, M <= 2^20. Otherwise MNB_ERR_INVALID_ARG or MNB_ERR_UNSUPPORTED.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream)
 *     and runs asynchronously: the call neither synchronises nor copies to the host,
 *     so every compute call may be captured into a CUDA graph. Launch geometry depends
 *     only on the shape arguments and the device.
 *   - Errors never throw. A non-MNB_OK status leaves a message for mnb_last_error()
 *     (per host thread). MNB_ERR_CUDA carries the CUDA error string.
 *   - Results are deterministic: the same inputs give the same bits on every run.
 */
#ifndef MNB_H_
#define MNB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MNB_API __attribute__((visibility("default")))
#else
#define MNB_API
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *mnb_stream;

typedef enum {
    MNB_OK = 0,
    MNB_ERR_INVALID_ARG = 1,  /* bad shape, block size, NULL pointer, or dtype */
    MNB_ERR_UNSUPPORTED = 2,  /* valid for the format, but not handled by this build */
    MNB_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    MNB_ERR_CAPTURE = 4,      /* the call is refused while `stream` is being captured */
    MNB_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
    MNB_ERR_TIMEOUT = 6       /* a bounded device-side wait gave up (kernel status word) */
} mnb_status;

typedef enum { MNB_F16 = 0, MNB_F32 = 1 } mnb_dtype;

/* One quantised weight: the MatMulNBits tuple (packed, scales, zero_points). */
typedef struct {
    const uint8_t *packed;      /* [N, K/2] bytes                                   */
    const void *scales;         /* [N, K/bs] of fp16 or fp32 (scales_dtype)          */
    int32_t scales_dtype;       /* MNB_F16 or MNB_F32                                */
    const uint8_t *zero_points; /* [N, ceil(K/bs/2)] nibbles, or NULL for zp = 8      */
} mnb_weight;

/*
 * Dequantise to fp32 [K, N] (row k, column n at out_kn[k*N + n]).
 * Follows matmul_nbits_dequant_f32 (matmul_nbits.rs): element (code - zp) * scale.
 * The product is rounded once to fp32 (round to nearest even); it is exact for fp16
 * scales. out_kn holds K*N floats.
 */
MNB_API mnb_status mnb_dequant(mnb_weight w, int K, int N, int block_size, float *out_kn,
                       mnb_stream stream);

/*
 * Size in bytes of the repacked tensor-core operand for a K x N weight:
 * ceil(N/128)*128 * ceil(K/64)*64 / 2. Returns 0 for invalid arguments.
 */
MNB_API size_t mnb_repacked_bytes(int K, int N, int block_size);

/*
 * Reorder `packed` into this library's tensor-core operand layout (a bijection on the
 * codes; scales and zero points keep their MatMulNBits indexing). The pages repack
 * once for their mma.sync kernel (marlin_gemm.rs, "Repacked weight layout"); the layout
 * here is new, built for 1-D bulk copies and shared-memory dequantisation:
 *   tile t (128 rows) and k-block b (64 k) form one 4096-byte block at
 *   (t * ceil(K/64) + b) * 4096; in it the 16 bytes at q*2048 + r*16 (q in 0..1,
 *   r in 0..127) hold the codes of row n = 128t + r for k = 64b + 32q + i, i in 0..31,
 *   as four little-endian 32-bit words; word j = i/8 keeps i at nibble p (bits 4p..4p+3)
 *   where i = 8j + 2(p%4) + p/4. Codes outside the K x N weight are 0.
 * `out` holds mnb_repacked_bytes(K, N, block_size) bytes. Runs once per weight, so it is
 * refused with MNB_ERR_CAPTURE while `stream` is capturing (a repack inside a graph
 * would be replayed on every launch).
 */
MNB_API mnb_status mnb_repack(const uint8_t *packed, int K, int N, int block_size, uint8_t *out,
                      mnb_stream stream);

/*
 * Decode GEMV, M = 1: Y[n] = sum_k A[k] * dequant(B)[n, k], stored as fp16 (round to
 * nearest even from the fp32 accumulator). A is fp16 [K], Y is fp16 [N].
 * The per-group partial dot of (code - zp) and A is scaled after it is formed
 * (matmul_nbits.rs, matmul_nbits_gemv_f16; marlin_gemm.rs, "Per-group scale applied
 * after the tensor-core accumulate"). |Y - exact| <= 2e-3 * sum_k |a_k w_nk| + 1e-5.
 */
MNB_API mnb_status mnb_gemv(const void *A, mnb_weight w, int K, int N, int block_size, void *Y,
                    mnb_stream stream);

/*
 * Scratch bytes for mnb_gemm (and mnb_gemm_bias) at this shape (0 when none): fp32
 * partials ([slices, M, N]) of a K split, summed in slice order, so results stay
 * deterministic.
 *   2 <= M <= 16: required when K is too large for one shared-memory pass of the small-M
 *   kernel; the size is an upper bound over the scale dtype and zero points.
 *   M > 16: optional; with it, outputs with fewer 128 x 256 tiles than half the SMs split
 *   K (whole quant groups) over the SMs, without it they run unsplit. The size covers
 *   GPUs of up to 160 SMs.
 * The caller allocates it once and passes it to every call of that shape; its contents
 * need no initialisation, each call overwrites them, so calls sharing one workspace must
 * be ordered on one stream.
 */
MNB_API size_t mnb_workspace_bytes(int M, int K, int N, int block_size);

/*
 * Y[M, N] = A[M, K] . dequant(B)^T, fp16 in and out, fp32 accumulation.
 * M = 1 runs the GEMV. 2 <= M <= 16 (speculative verify) streams the MatMulNBits
 * storage directly; `repacked` may be NULL and is not read. M > 16 needs the repacked
 * operand from mnb_repack (`repacked` NULL gives MNB_ERR_INVALID_ARG) and runs on the
 * tcgen05 tensor cores,
 * the group scale applied to each group's partial accumulator (marlin_gemm.rs,
 * matmul_nbits_marlin_gemm_f16). `workspace`/`ws_bytes`: see mnb_workspace_bytes;
 * for 2 <= M <= 16 a smaller workspace gives MNB_ERR_INVALID_ARG.
 */
MNB_API mnb_status mnb_gemm(const void *A, int M, mnb_weight w, const uint8_t *repacked, int K, int N,
                    int block_size, void *workspace, size_t ws_bytes, void *Y,
                    mnb_stream stream);

/* Bias epilogue modes for mnb_gemm_bias. */
typedef enum {
    MNB_BIAS_NONE = 0,         /* Y = fp16(acc)                                          */
    MNB_BIAS_FUSED = 1,        /* Y = fp16(acc + b), one rounding (a fused MatMul+bias)   */
    MNB_BIAS_AFTER_ROUND = 2   /* Y = fp16(fp16(acc) + b), bit-identical to mnb_gemm
                                  followed by a separate fp16 add                          */
} mnb_bias_mode;

/*
 * mnb_gemm with a bias [N] (fp16, one value per output column) added in the epilogue,
 * in either of the two rounding orders of the pages' fp16 bias epilogue (matmul_nbits.rs,
 * fold_bias_f16; marlin_gemm.rs, fold_bias): MNB_BIAS_FUSED adds b to the fp32
 * accumulator and rounds once, MNB_BIAS_AFTER_ROUND rounds the accumulator to fp16 first
 * and then rounds fp32(that) + b. `bias` may be NULL only with MNB_BIAS_NONE.
 */
MNB_API mnb_status mnb_gemm_bias(const void *A, int M, mnb_weight w, const uint8_t *repacked, int K,
                                 int N, int block_size, const void *bias, int bias_mode,
                                 void *workspace, size_t ws_bytes, void *Y, mnb_stream stream);

/*
 * Paired gate/up projection with the SwiGLU epilogue (matmul_nbits.rs,
 * matmul_nbits_gemv_f16_gate_up_swiglu): g = A . gate^T, u = A . up^T (both M = 1,
 * same K, N, block_size), out[n] = silu(g[n]) * u[n] with silu(x) = x / (1 + e^-x),
 * computed in fp32 from the fp32 accumulators and stored as fp16. A is fp16 [K],
 * out is fp16 [N]. Each weight may use its own scale dtype and zero points.
 */
MNB_API mnb_status mnb_gemv_gate_up_swiglu(const void *A, mnb_weight gate, mnb_weight up, int K, int N,
                                   int block_size, void *out, mnb_stream stream);

/*
 * ---- fp32 activations ----
 *
 * The operator's fp32 path (matmul_nbits.rs, MatMulNBitsKernel::run with a Float32 A:
 * matmul_nbits_gemv_f32 for M = 1, dequantise-then-GEMM otherwise): A [M, K], Y [M, N]
 * and the optional bias [N] are fp32 (row-major, 16-byte aligned), Y = A . dequant(B)^T
 * + bias with no fp16 rounding anywhere. M = 1 multiplies fp32 activations directly. For
 * M >= 2 every row of A is scaled by a power of two and split into two fp16 rows (high
 * and low part, together within 2^-22 of the row) that the fp16 tensor-core kernels
 * multiply; their two accumulators are added and scaled back in fp32. Either way the
 * weights are exact and the accumulation is fp32, so |Y - exact| <= 2e-3 * sum_k |a_k
 * w_nk| + 1e-5 holds with a wide margin. A row holding inf or NaN gives non-finite
 * outputs in that row.
 */

/*
 * Workspace bytes for mnb_gemm_f32: 0 for M = 1, else 4*M*K (the split activation) +
 * 4*M rounded up to 16 (row exponents) + mnb_workspace_bytes(2*M, K, N, block_size)
 * (the K-slice partials of the 2*M split rows: required for M <= 8, optional above, as
 * in mnb_gemm).
 */
MNB_API size_t mnb_workspace_bytes_f32(int M, int K, int N, int block_size);

/*
 * fp32 Y[M, N] = A[M, K] . dequant(B)^T (+ bias[n] when bias is not NULL). Weight
 * arguments as mnb_gemm; `repacked` (mnb_repack) is required when M > 8, because the
 * split activation then has more than 16 rows and runs on the tcgen05 kernel. The
 * workspace holds the split activation, the row exponents and any K-slice partials; its contents need no
 * initialisation and are overwritten by each call, so calls sharing one workspace must
 * be ordered on one stream.
 */
MNB_API mnb_status mnb_gemm_f32(const float *A, int M, mnb_weight w, const uint8_t *repacked, int K, int N,
                                int block_size, const float *bias, void *workspace, size_t ws_bytes, float *Y,
                                mnb_stream stream);

/*
 * ---- Act-order weights (g_idx) ----
 *
 * MatMulNBits takes an optional int32 group index g_idx[K] (matmul_nbits.rs,
 * MatMulNBitsKernel::run, input 4; kernel matmul_nbits_dequant_f32): the scale and zero
 * point of column k are those of group g_idx[k] instead of group k / bs, while the code
 * still sits in block k / bs:
 *   dequant(B)[n, k] = (code[n, k] - zp[n, g_idx[k]]) * scale[n, g_idx[k]].
 * The pages check every entry with a device-to-host copy on each call. Here the check
 * happens once, on the host, when the weight is prepared (mnb_act_order_plan), and the
 * weight is rewritten into an equivalent plain block weight of K' columns
 * (mnb_act_order_prepare): k sorted by group, ascending k inside a group, each group's
 * run padded with empty slots to whole blocks. Each call then gathers the activation
 * into the same order and runs the ordinary kernels, so every per-call entry point
 * below is capture-safe. With g_idx[k] = k / bs the prepared weight is the original.
 */

/*
 * Dequantise with a group index per k to fp32 [K, N] (out_kn[k*N + n]), as
 * matmul_nbits_dequant_f32 does when given group indices: element
 * (code[n, k] - zp[n, g]) * scale[n, g], g = g_idx[k], rounded once to fp32. g_idx is
 * device int32 [K]. An entry outside 0..K/bs-1 writes 0 for that k (the pages' kernel
 * rule) and sets the index bit of the device status word, which mnb_check_device_status
 * reports as MNB_ERR_INVALID_ARG.
 */
MNB_API mnb_status mnb_dequant_gidx(mnb_weight w, const int32_t *g_idx, int K, int N, int block_size,
                                    float *out_kn, mnb_stream stream);

/*
 * Host-only planning step (no GPU work). g_idx is HOST int32 [K]; every entry must lie
 * in 0..K/bs-1, else MNB_ERR_INVALID_ARG names the first bad entry (the operator's own
 * check, matmul_nbits.rs). Writes *K_prepared = K' = bs * sum_g ceil(count_g / bs), with
 * K <= K' <= 2K (K' = K when every group has exactly bs members, the act-order
 * quantisation case). If perm is not NULL it receives K' entries (host int32): perm[k']
 * = the source column of prepared column k', or -1 for an empty slot. If block_group is
 * not NULL it receives K'/bs entries: the group of each prepared block. Call once with
 * NULL arrays to learn K', or size both for the 2K worst case.
 */
MNB_API mnb_status mnb_act_order_plan(const int32_t *g_idx, int K, int block_size, int32_t *K_prepared,
                                      int32_t *perm, int32_t *block_group);

/*
 * Write the prepared weight (device buffers owned by the caller, same block_size, K'
 * columns): packed_out [N, K'/2] bytes with codes code[n, perm[k']] (the block's zero
 * point at an empty slot, so its weight is 0); scales_out [N, K'/bs] of w.scales_dtype,
 * scales_out[n, j] = scales[n, block_group[j]]; zero_points_out [N, ceil(K'/bs/2)] bytes
 * (nibbles as in MatMulNBits, the unused high nibble of an odd count 0), required when w
 * has zero points and ignored otherwise (the prepared weight then has none either).
 * perm [K'] and block_group [K'/bs] are device copies of mnb_act_order_plan's output.
 * For M > 16 repack packed_out with mnb_repack(packed_out, K', N, block_size, ...).
 * Runs once per weight, so it is refused with MNB_ERR_CAPTURE while `stream` captures.
 */
MNB_API mnb_status mnb_act_order_prepare(mnb_weight w, int K, int N, int block_size, const int32_t *perm,
                                         const int32_t *block_group, int K_prepared, uint8_t *packed_out,
                                         void *scales_out, uint8_t *zero_points_out, mnb_stream stream);

/*
 * A_out[m, k'] = A[m, perm[k']] for m < M, k' < K', and +0 where perm[k'] = -1 (fp16,
 * row-major; A is [M, K], A_out is [M, K']). perm is device int32 [K'] and K' a
 * multiple of 8 no larger than 2K. Any other perm entry writes 0 and sets the index
 * bit of the device status word.
 */
MNB_API mnb_status mnb_act_order_gather(const void *A, int M, int K, const int32_t *perm, int K_prepared,
                                        void *A_out, mnb_stream stream);

/* Workspace bytes mnb_gemm_act_order needs: M * K' * 2 (the gathered activation). */
MNB_API size_t mnb_act_order_workspace_bytes(int M, int K_prepared);

/*
 * Y[M, N] = A[M, K] . dequant_g_idx(B)^T for an act-order weight, with the bias modes of
 * mnb_gemm_bias. `w` and `repacked` are the PREPARED weight (K' columns; `repacked`
 * needed for M > 16 as in mnb_gemm); perm is the device copy of the plan's perm. The call
 * gathers A into `workspace` (at least mnb_act_order_workspace_bytes(M, K') bytes,
 * contents need no initialisation, overwritten by each call) and then runs mnb_gemm's
 * kernel for (M, K', N) on it. A workspace larger by at least
 * mnb_workspace_bytes(M, K', N, block_size), placed after the gathered activation rounded
 * up to 16 bytes, lets 2 <= M <= 16 with K' beyond one shared-memory pass run on the
 * small-M kernel's K slices (without it those calls take the generic kernel). Calls that
 * share one workspace must be ordered on one stream. Tolerance as mnb_gemm, with the bound
 * taken over the g_idx weights.
 */
MNB_API mnb_status mnb_gemm_act_order(const void *A, int M, mnb_weight w, const uint8_t *repacked,
                                      const int32_t *perm, int K, int K_prepared, int N, int block_size,
                                      const void *bias, int bias_mode, void *workspace, size_t ws_bytes,
                                      void *Y, mnb_stream stream);

/*
 * mnb_gemm_act_order without a workspace, for callers that cannot allocate device
 * memory (a plugin inside a host framework that owns all device memory and hands it no
 * workspace, or a loop where cudaMalloc's implicit synchronisation is not allowed). The
 * published MatMulNBits descriptions have no counterpart: this entry point is this
 * library's own.
 * Same arguments and result as mnb_gemm_act_order minus workspace/ws_bytes. The
 * gathered activation (M * K' * 2 bytes) lives in a static device array of 8 MiB
 * (8388608 bytes) inside the library, held on every GPU that loads the library until
 * the process exits; a larger M * K' gives MNB_ERR_UNSUPPORTED. The call allocates
 * nothing. Its first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture. All calls share the one array and it keeps the last call's contents
 * (each call overwrites everything it reads, so nothing needs clearing): calls that
 * may overlap on the GPU (different streams, or threads without ordering) race on it,
 * so order them on one stream.
 */
MNB_API mnb_status mnb_gemm_act_order_noalloc(const void *A, int M, mnb_weight w, const uint8_t *repacked,
                                              const int32_t *perm, int K, int K_prepared, int N,
                                              int block_size, const void *bias, int bias_mode, void *Y,
                                              mnb_stream stream);

/*
 * Programmatic dependent launch. With `enable` != 0, later calls on this host thread
 * launch their kernels with programmatic stream serialisation: a kernel may start while
 * the previous kernel on the stream is still running, and it streams its weight, scale
 * and zero-point buffers (and an act-order perm) before waiting for that kernel to
 * finish; it reads A and writes Y only after the wait. Enable it only when no earlier
 * work on the stream writes those buffers (weights that stay constant during
 * inference). Default: off.
 */
MNB_API void mnb_set_programmatic_launch(int enable);

/*
 * Reads and clears the device status word. Kernels that wait on shared-memory barriers
 * bound every wait; one that gives up sets a bit in this word, writes NaN outputs and
 * returns instead of hanging. The act-order kernels set another bit for an index input
 * out of range. Returns MNB_ERR_TIMEOUT (with the bits in the message) if a wait gave
 * up, MNB_ERR_INVALID_ARG if only the index bit is set, else MNB_OK. Synchronises the
 * current device, so it must not be called while a stream is being captured.
 */
MNB_API mnb_status mnb_check_device_status(void);

/*
 * Self-test of the failure path above (no counterpart on the pages; the bounded waits are
 * this library's own): launches one kernel on `stream` whose bounded wait on a
 * shared-memory barrier that nothing ever arrives on gives up after `limit_us`
 * microseconds (1 .. 1000000, else MNB_ERR_INVALID_ARG), sets the wait bit of the device
 * status word and returns. Nothing faults and the context stays usable; the next
 * mnb_check_device_status returns MNB_ERR_TIMEOUT and clears the word. For tests.
 */
MNB_API mnb_status mnb_selftest_wait_timeout(unsigned int limit_us, mnb_stream stream);

/* Message of the last failed call on this host thread ("" if none). */
MNB_API const char *mnb_last_error(void);

/* Name of the kernel variant the last successful call on this host thread launched. */
MNB_API const char *mnb_last_variant(void);

/* Library version string. */
MNB_API const char *mnb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MNB_H_ */
