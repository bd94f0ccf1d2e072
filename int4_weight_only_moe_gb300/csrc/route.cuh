// Router arithmetic shared by the router kernel and the small-batch routing +
// gather kernel: renormalised top-k softmax over one token's router logits (the
// gating network that picks which experts' weights a token needs, "The
// Weight-Streaming Threshold", Input Knowledge Required): the k largest logits in
// descending order, equal logits by ascending expert id, with weights
// exp(l_j - l_max) / sum over the k selected of exp(l_i - l_max) -- the softmax
// over all experts restricted to the selected ones and renormalised.
#pragma once
#include <climits>
#include <cmath>
#include <cstdint>

namespace moe {

// Top-k of one token's logits row by one warp. Lane l holds experts l, l + 32,
// ... (at most 32 each, E <= 1024); every round each lane offers its best untaken
// expert and a butterfly reduction picks the warp's best (larger logit, then the
// lower id). Lane j < k receives the j-th winner and its renormalised weight.
// NaN logits rank as -infinity.
__device__ __forceinline__ void warp_topk(const float* __restrict__ row, int E, int k, int lane, int* win_id,
                          float* win_w) {
  float v[32];
  const int nslots = (E + 31) >> 5;
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = i * 32 + lane;
    float x = -INFINITY;
    if (i < nslots && e < E) {
      x = row[e];
      if (x != x) x = -INFINITY;
    } else {
      taken |= 1u << i;
    }
    v[i] = x;
  }
  float my_v = -INFINITY;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i >= nslots) break;
      if (!((taken >> i) & 1u) && (bi < 0 || v[i] > bv)) {
        bv = v[i];
        bi = i;
      }
    }
    int be = bi >= 0 ? bi * 32 + lane : INT_MAX;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be != INT_MAX && lane == (be & 31)) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const float p = lane < k ? expf(my_v - top) : 0.0f;
  float z = p;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  *win_id = my_e;
  *win_w = p / z;
}

}  // namespace moe
