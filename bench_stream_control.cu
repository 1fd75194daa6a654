// Streaming-only control for the M = 1 GEMV (a measurement instrument beside bench.py; not
// part of the library).
//
// It moves exactly the bytes the tensor-core GEMV moves for the attention-projection shape
// (K = N = 4096, block size 32, fp16 scales, zero points) with the same launch structure --
// one CTA of 8 consumer warps and 1 producer warp per SM, two CTAs resident per SM, all of a
// CTA's stages requested before the programmatic-launch wait, 1000 calls in one CUDA graph
// with programmatic dependent launch, weight copies rotated through HBM -- and does no
// arithmetic: after the wait the consumers read the activation, wait for every stage, and
// each tile's last warp stores 16 zeros.  The time per call is the floor of that launch and
// copy structure; the GEMV's time above it is its compute.
//
// Build and run (bench.py --stream-control does both):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 -I gemm_mnb_gemv_gb300/csrc \
//        bench_stream_control.cu -o _build/stream_control && _build/stream_control
// Prints one JSON object.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <vector>

#include "mnb_device.cuh"
#include "tcgen05.cuh"

namespace {

constexpr int kRows = 16, kBox = 2048, kMaxStages = 8, kNcw = 8;
constexpr int K = 4096, N = 4096, BS = 32, G = K / BS, SROW = G * 2, ZROW = G / 2;

struct Args {
  const __half* A;
  const uint8_t* zp;
  __half* Y;
  int ntiles, stages, stage_bytes, poff, zoff;
};

__global__ void __launch_bounds__((kNcw + 1) * 32, 2)
    stream_kernel(const Args p, const __grid_constant__ CUtensorMap tp, const __grid_constant__ CUtensorMap ts) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStages];
  __shared__ unsigned cnt[kMaxStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = mnb::smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int t0 = (int)(((long long)blockIdx.x * p.ntiles) / gridDim.x);
  const int t1 = (int)(((long long)(blockIdx.x + 1) * p.ntiles) / gridDim.x);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mnb::mbar_init(&full_bar[s], 1);
      cnt[s] = 0;
    }
    mnb::fence_mbar_init();
  }
  __syncthreads();
  if (warp == kNcw) {
    if (lane == 0)
      for (int i = 0; i < t1 - t0; ++i) {
        uint8_t* wb = ring + (size_t)i * p.stage_bytes;
        const int n0 = (t0 + i) * kRows;
        mnb::mbar_arrive_expect_tx(&full_bar[i], (uint32_t)((16 + 2) * kBox + kRows * ZROW));
        mnb::tc::tma_load_3d(wb + p.poff, &tp, 0, n0, 0, &full_bar[i]);
        mnb::tc::tma_load_3d(wb, &ts, 0, n0, 0, &full_bar[i]);
        mnb::bulk_g2s(wb + p.zoff, p.zp + (long long)n0 * ZROW, kRows * ZROW, &full_bar[i]);
      }
    __syncwarp();
    if (lane == 0)
      for (int i = 0; i < t1 - t0; ++i) (void)mnb::mbar_wait_bounded(&full_bar[i], 0);
    mnb::pdl_launch_dependents();
  } else {
    mnb::pdl_launch_dependents();
    mnb::pdl_wait();
    // the activation read each warp does in the GEMV (its blocks of A)
    const uint4 x = *reinterpret_cast<const uint4*>(p.A + (warp * 2) * 256 + 8 * lane);
    for (int i = 0; i < t1 - t0; ++i) {
      (void)mnb::mbar_wait_bounded(&full_bar[i], 0);
      __syncwarp();
      unsigned last = 0;
      if (lane == 0) last = atomicInc(&cnt[i], kNcw - 1) == kNcw - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last && lane < kRows) {
        const int n = (t0 + i) * kRows + lane;
        if (n < N) p.Y[n] = __ushort_as_half((unsigned short)((x.x & 0) + (x.w & 0)));
      }
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  cudaDriverEntryPointQueryResult q;
  void* f = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

#define CHECK(x)                                                                  \
  do {                                                                            \
    cudaError_t e_ = (x);                                                         \
    if (e_ != cudaSuccess) {                                                      \
      printf("{\"error\": \"%s at line %d\"}\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                                   \
    }                                                                             \
  } while (0)

}  // namespace

int main() {
  int sms = 0;
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  auto encode = encode_fn();
  if (!encode) {
    printf("{\"error\": \"no cuTensorMapEncodeTiled\"}\n");
    return 1;
  }
  const size_t pbytes = (size_t)N * K / 2, sbytes = (size_t)N * SROW, zbytes = (size_t)N * ZROW;
  const size_t per_copy = pbytes + sbytes + zbytes;
  const int copies = (int)((3ull * 126 * 1024 * 1024) / per_copy + 2);
  std::vector<uint8_t*> P(copies), S(copies), Z(copies);
  for (int c = 0; c < copies; ++c) {
    CHECK(cudaMalloc(&P[c], pbytes));
    CHECK(cudaMalloc(&S[c], sbytes));
    CHECK(cudaMalloc(&Z[c], zbytes));
    CHECK(cudaMemset(P[c], 0x11, pbytes));
    CHECK(cudaMemset(S[c], 0x22, sbytes));
    CHECK(cudaMemset(Z[c], 0x88, zbytes));
  }
  __half *A, *Y;
  CHECK(cudaMalloc(&A, K * 2));
  CHECK(cudaMalloc(&Y, N * 2));
  CHECK(cudaMemset(A, 0, K * 2));
  const int ntiles = N / kRows, grid = sms < ntiles ? sms : ntiles;
  const int max_tiles = (ntiles + grid - 1) / grid;
  Args a;
  a.A = A;
  a.Y = Y;
  a.ntiles = ntiles;
  a.stages = max_tiles;
  a.poff = 2 * kBox;                 // two scale boxes (256 bytes of fp16 scales per row)
  a.zoff = a.poff + 16 * kBox;       // 16 packed segments (2 KB per row)
  a.stage_bytes = (a.zoff + kRows * ZROW + 1023) / 1024 * 1024;
  const size_t smem = (size_t)a.stages * a.stage_bytes + 1024;
  CHECK(cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  std::vector<CUtensorMap> tp(copies), ts(copies);
  for (int c = 0; c < copies; ++c) {
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t pdim[3] = {128, N, K / 256}, pstr[2] = {K / 2, 128};
    const cuuint32_t pbox[3] = {128, kRows, 16};
    const cuuint64_t sdim[3] = {128, N, SROW / 128}, sstr[2] = {SROW, 128};
    const cuuint32_t sbox[3] = {128, kRows, SROW / 128};
    if (encode(&tp[c], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, P[c], pdim, pstr, pbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ||
        encode(&ts[c], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, S[c], sdim, sstr, sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) {
      printf("{\"error\": \"tensor map\"}\n");
      return 1;
    }
  }
  cudaStream_t st;
  CHECK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  auto launch = [&](int c) {
    a.zp = Z[c];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((kNcw + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stream_kernel, a, tp[c], ts[c]);
  };
  const int calls = 1000;
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  CHECK(cudaStreamBeginCapture(st, cudaStreamCaptureModeGlobal));
  for (int i = 0; i < calls; ++i) CHECK(launch(i % copies));
  CHECK(cudaStreamEndCapture(st, &graph));
  CHECK(cudaGraphInstantiate(&exec, graph, 0));
  for (int w = 0; w < 5; ++w) CHECK(cudaGraphLaunch(exec, st));
  CHECK(cudaStreamSynchronize(st));
  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  const int reps = 20;
  CHECK(cudaEventRecord(e0, st));
  for (int r = 0; r < reps; ++r) CHECK(cudaGraphLaunch(exec, st));
  CHECK(cudaEventRecord(e1, st));
  CHECK(cudaEventSynchronize(e1));
  float ms = 0;
  CHECK(cudaEventElapsedTime(&ms, e0, e1));
  const double us = ms * 1e3 / (reps * calls);
  const double bytes = (double)per_copy + 2.0 * K + 2.0 * N;
  printf("{\"workload\": \"gemv_attnproj_k4096_n4096 streaming-only control\", \"us_per_call\": %.4f, "
         "\"gbps\": %.1f, \"copies\": %d, \"calls_per_replay\": %d, \"ctas\": %d, \"stages_per_cta\": %d}\n",
         us, bytes / (us * 1e3), copies, calls, grid, a.stages);
  return 0;
}
