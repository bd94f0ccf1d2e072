// Allocation-free forward: moe_w4a16_forward with its scratch workspace in a
// fixed array of the library's device image instead of caller-provided memory,
// for callers that cannot allocate device memory themselves.
#include <cuda.h>

#include <mutex>
#include <string>

#include "../../include/moe_w4a16.h"
#include "kernels.cuh"

namespace moe {
int report_error(int code, const char* msg);
}

namespace {

constexpr size_t kNoAllocBytes = MOE_W4A16_NOALLOC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The scratch of every allocation-free call on a device. In host code this name
// is only a host-side stand-in: its device address comes from
// cudaGetSymbolAddress, with the device current.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocBytes];

// Per device: the array's address and the id of the CUDA context it was looked
// up in. A device reset (cudaDeviceReset) or a re-created primary context loads
// the library's device image afresh, and the array can move; the context id
// (unique for the life of the process) tells a stale address from a valid one.
struct Cached {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
  bool valid = false;
};
std::mutex g_noalloc_mutex;
Cached g_noalloc[kMaxDevices];

// Driver entry points for the current context's id, fetched through the runtime
// (the library does not link the driver library directly).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_entry_points_tried = false;

// Id of the calling thread's current context, or 0 when it cannot be read (then
// the address is looked up again on every call).
unsigned long long current_context_id() {
  if (!g_entry_points_tried) {
    g_entry_points_tried = true;
    cudaDriverEntryPointQueryResult q1{}, q2{};
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    } else {
      cudaGetLastError();
    }
  }
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

}  // namespace

extern "C" int moe_w4a16_forward_noalloc(moe_w4a16_t h, const uint16_t* hidden,
                                         const int32_t* topk_ids, const float* topk_weights,
                                         uint16_t* out, int M, void* stream) {
  if (!h) return moe::report_error(MOE_W4A16_INVALID_ARG, "null handle");
  if (M < 0) return moe::report_error(MOE_W4A16_INVALID_ARG, "M must be >= 0");
  const size_t need = moe_w4a16_workspace_size(h, M);
  if (need > kNoAllocBytes) {
    const std::string msg = "allocation-free forward: M=" + std::to_string(M) + " needs " +
                            std::to_string(need) + " bytes of workspace, the static array holds " +
                            std::to_string(kNoAllocBytes) + " bytes";
    return moe::report_error(MOE_W4A16_WORKSPACE_TOO_SMALL, msg.c_str());
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return moe::report_error(MOE_W4A16_CUDA_ERROR,
                             (std::string("cudaGetDevice: ") + cudaGetErrorString(e)).c_str());
  if (dev < 0 || dev >= kMaxDevices)
    return moe::report_error(MOE_W4A16_UNSUPPORTED_SHAPE, "device index beyond 63");
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const unsigned long long ctx = current_context_id();
    Cached& c = g_noalloc[dev];
    if (!c.valid || ctx == 0 || c.ctx_id != ctx) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
      if (e != cudaSuccess || !p) {
        c.valid = false;
        return moe::report_error(
            MOE_W4A16_CUDA_ERROR,
            (std::string("cudaGetSymbolAddress(static workspace): ") + cudaGetErrorString(e)).c_str());
      }
      c.ptr = p;
      // the lookup made the device's context current if it was not yet
      c.ctx_id = ctx != 0 ? ctx : current_context_id();
      c.valid = c.ctx_id != 0;
    }
    ws = c.ptr;
  }
  return moe_w4a16_forward(h, hidden, topk_ids, topk_weights, out, M, ws, kNoAllocBytes, stream);
}
