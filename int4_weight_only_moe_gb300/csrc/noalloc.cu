// Allocation-free forward: moe_w4a16_forward with its scratch workspace in a
// fixed array of the library's device image instead of caller-provided memory,
// for callers that cannot allocate device memory themselves.
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
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

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
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
      if (e != cudaSuccess || !p)
        return moe::report_error(
            MOE_W4A16_CUDA_ERROR,
            (std::string("cudaGetSymbolAddress(static workspace): ") + cudaGetErrorString(e)).c_str());
      g_noalloc_ptr[dev] = p;
    }
    ws = g_noalloc_ptr[dev];
  }
  return moe_w4a16_forward(h, hidden, topk_ids, topk_weights, out, M, ws, kNoAllocBytes, stream);
}
