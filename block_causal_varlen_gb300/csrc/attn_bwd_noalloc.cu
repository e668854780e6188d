// Backward entry point that allocates nothing.
//
// Some callers cannot hand the library a device workspace: for example a
// plugin running inside another runtime that owns every device allocation
// and gives its plugins no allocator, or a caller under a hard device-memory
// cap where an extra allocation would fail. bd_attn_bwd_noalloc serves them:
// it runs the same backward as bd_attn_bwd with the workspace taken from a
// fixed array in device global memory that this file declares, so it calls
// no cudaMalloc / cudaFree and no allocating library routine.
//
// Costs and rules of that choice:
//   * every GPU that loads the library holds kScratchBytes for the array until
//     the process exits;
//   * plans whose workspace exceeds kScratchBytes are rejected (BD_ERR_CAPACITY)
//     before anything is launched;
//   * every call shares the one array per device, so calls that overlap on the
//     GPU (different streams without ordering between them) race on it;
//     callers must order such calls. A call fully rewrites the part of the
//     array it reads, so nothing has to start at zero;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current); make that first call
//     before any stream capture. The address is kept for the life of the
//     process, so a cudaDeviceReset (or any other teardown of the device's
//     context) between calls is not supported: the array may then sit at a new
//     address and the kept one would be stale.
#include <cuda_runtime.h>

#include <mutex>

#include "host_util.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB

// The host-side name of this array is only a stand-in: device code may use it
// directly, host code must use the address cudaGetSymbolAddress returns.
__device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

int32_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return bd::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return bd::fail(BD_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || !p) return bd::cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return BD_OK;
}

}  // namespace

extern "C" int32_t bd_attn_bwd_noalloc(const void* plan_host, const void* plan_dev, const bd_tensor* q,
                                       const bd_tensor* k, const bd_tensor* v, const bd_tensor* out,
                                       const bd_tensor* dout, const bd_rowstat* lse, bd_tensor* dq,
                                       bd_tensor* dk, bd_tensor* dv, int32_t accumulate_dkv, void* stream) {
  size_t need = 0;
  int32_t st = bd_attn_bwd_workspace(plan_host, &need);
  if (st) return st;
  if (need > kScratchBytes)
    return bd::fail(BD_ERR_CAPACITY, "plan needs %zu bytes of workspace; the fixed scratch holds %zu", need,
                    kScratchBytes);
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch))) return st;
  return bd_attn_bwd(plan_host, plan_dev, q, k, v, out, dout, lse, dq, dk, dv, accumulate_dkv, scratch,
                     kScratchBytes, stream);
}

extern "C" size_t bd_attn_bwd_noalloc_capacity(void) { return kScratchBytes; }
