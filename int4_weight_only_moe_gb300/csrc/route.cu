// Router kernel: top-k routing of every token's router logits (the arithmetic is
// in route.cuh), one warp per token.
#include "kernels.cuh"
#include "route.cuh"

namespace moe {

// One warp per token, grid-stride.
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int M, int E,
                                                    int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long t = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < M;
       t += nwarps) {
    int id;
    float w;
    warp_topk(logits + t * E, E, k, lane, &id, &w);
    if (lane < k) {
      ids[t * k + lane] = id;
      wts[t * k + lane] = w;
    }
  }
  pdl_launch_dependents();
}

cudaError_t launch_route(const float* logits, int M, int E, int k, int32_t* ids, float* wts,
                         int num_sms, cudaStream_t stream, bool pdl) {
  if (M <= 0) return cudaSuccess;
  long long grid = (static_cast<long long>(M) + 7) / 8;
  const long long cap = 8LL * num_sms;
  if (grid > cap) grid = cap;
  return launch_k(route_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream, pdl, logits, M,
                  E, k, ids, wts);
}

}  // namespace moe
