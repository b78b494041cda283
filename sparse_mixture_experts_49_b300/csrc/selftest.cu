// Self-test of the bounded on-chip waits. Every mbarrier wait in the
// library's kernels gives up after a fixed time without progress, records
// MOE_DEVERR_TIMEOUT in the workspace's error word and lets its kernel
// return, so that a broken handshake costs an error code instead of a hung
// GPU. This entry point runs that same wait, with the same limit, on a
// barrier that nothing completes: one thread of one block waits, gives up,
// records the error and the block exits.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_probe_kernel(DeviceStatus *st) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // phase 0 needs one arrival, which never comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) (void)mbar_wait_bounded(&bar, 0, &abort_flag, st);
}

}  // namespace

}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(void *ws, moe_stream_t stream) {
  using namespace moe;
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return MOE_ERR_ALIGNMENT;
  // the error word is the first bytes of every workspace
  cudaError_t e = launch_kernel(bounded_wait_probe_kernel, dim3(1), dim3(32), 0, (cudaStream_t)stream,
                                static_cast<DeviceStatus *>(ws));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
