// moe_dispatch_noalloc: the dispatch of moe_dispatch for callers that cannot
// give the library any scratch memory.
//
// Some callers cannot allocate device memory at all: a plugin running inside
// a host framework that owns every device allocation, or a latency-critical
// path that cannot pay for cudaMalloc's device-wide synchronisation. Such a
// caller has no workspace to pass. This entry point keeps the dispatch's
// scratch (per-block expert counts, their per-expert scan, the expert loads
// and an error word) in one fixed array compiled into the library, so the
// call itself allocates nothing. The caller still passes every input and
// output.
//
// Costs and limits of that choice:
//   - the array has a fixed size: T <= MOE_NOALLOC_MAX_TOKENS (32768) tokens
//     and E <= 256 experts, about 256 KB, and every GPU that loads the library
//     holds it until the process exits;
//   - the first call on a device (and the first after a device reset) looks
//     the array's address up with cudaGetSymbolAddress; that first call
//     should come before any stream capture;
//   - all calls share the array and it keeps the last call's contents: two
//     calls whose work can overlap on the GPU race with each other;
//   - bad or repeated expert indices are still treated as dropped, but the
//     error word is private to the library, so they are not reported.
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxBlocks = MOE_NOALLOC_MAX_TOKENS / DISPATCH_TOKENS;
constexpr int kMaxExperts = 256;
constexpr size_t kStatusInts = 64;  // keeps the count arrays 256-byte aligned
constexpr size_t kCountInts = (size_t)kMaxBlocks * kMaxExperts;
constexpr size_t kScratchInts = kStatusInts + 2 * kCountInts;
constexpr int kMaxDevices = 64;

// Layout (int32 units): [error word, completion counter | per-block counts | per-block bases].
static __device__ __align__(256) int32_t g_dispatch_scratch[kScratchInts];

std::mutex g_mutex;
int32_t *g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // unique id of the context the address belongs to

// Unique id of the calling thread's current CUDA context (0 if it cannot be
// read). A device reset destroys the primary context and the module loaded in
// it; the context created after it has a new id, so a cached address is never
// reused across a reset. Driver entry points are looked up at run time, so the
// library needs no link-time dependency on libcuda.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext *);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *a = nullptr, *b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<GetCurrentFn>(a);
      get_id = reinterpret_cast<GetIdFn>(b);
    }
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
      get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of g_dispatch_scratch on the current device, looked up once
// per device and context (set-up work: the first call on a device, or the
// first after a device reset, calls cudaGetSymbolAddress).
cudaError_t scratch_on_current_device(int32_t **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // 0 when no context is current yet: then the lookup below creates the
  // device's primary context, and the id is read again after it.
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr || ctx == 0 || g_scratch_ctx[dev] != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t *>(p);
    g_scratch_ctx[dev] = current_context_id();
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace moe

static moe_status dispatch_noalloc_impl(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                                           int32_t *slot, int32_t *kept, int32_t *expert_offsets,
                                           int32_t *row_token, void *x_perm, moe_stream_t stream) {
  using namespace moe;
  Shape sh;
  moe_status st = dispatch_shape(cfg, &sh);
  if (st != MOE_OK) return st;
  const void *ptrs[] = {x, topk_idx, slot, kept, expert_offsets, row_token, x_perm};
  for (const void *p : ptrs) {
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
  }
  if (sh.T > MOE_NOALLOC_MAX_TOKENS || sh.E > kMaxExperts || sh.reroute) return MOE_ERR_UNSUPPORTED;
  int32_t *base = nullptr;
  cudaError_t e = scratch_on_current_device(&base);
  if (e != cudaSuccess) return report_cuda(e);
  DeviceStatus *status = reinterpret_cast<DeviceStatus *>(base);
  int32_t *counts = base + kStatusInts;
  int32_t *bases = counts + kCountInts;
  unsigned int *counter = reinterpret_cast<unsigned int *>(base + 32);
  // Only the error word and the completion counter must start at zero; the
  // kernels overwrite everything else they read.
  e = cudaMemsetAsync(base, 0, kStatusInts * sizeof(int32_t), (cudaStream_t)stream);
  if (e != cudaSuccess) return report_cuda(e);
  return report_cuda(launch_dispatch_with_scratch(sh, x, topk_idx, slot, kept, expert_offsets, row_token, x_perm,
                                                  nullptr, counts, bases, counter, status, (cudaStream_t)stream));
}

extern "C" moe_status moe_dispatch_noalloc(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                                           int32_t *slot, int32_t *kept, int32_t *expert_offsets,
                                           int32_t *row_token, void *x_perm, moe_stream_t stream) {
  nvtxRangePushA("moe_dispatch_noalloc");  // NVTX range over the call (a no-op without a tool attached)
  const moe_status s = dispatch_noalloc_impl(cfg, x, topk_idx, slot, kept, expert_offsets, row_token, x_perm, stream);
  nvtxRangePop();
  return s;
}
