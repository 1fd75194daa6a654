// Self-test of the bounded device-side waits: a kernel that waits on an mbarrier nobody
// ever arrives on, with a short limit, so the wait gives up, records the timeout in the
// device status word and the kernel returns.  It faults nothing and leaves the context
// usable; mnb_check_device_status then reports MNB_ERR_TIMEOUT.
#include "mnb_device.cuh"
#include "mnb_internal.h"

namespace mnb {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none ever comes
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait_bounded_ns(&bar, 0u, limit_ns)) report_status(status, kStatusFullWait);
}

}  // namespace

cudaError_t launch_wait_selftest(LaunchCtx& ctx, uint64_t limit_ns) {
  ctx.variant = "wait_selftest";
  return launch_kernel(ctx, wait_selftest_kernel, dim3(1), dim3(32), 0, ctx.status, limit_ns);
}

}  // namespace mnb
