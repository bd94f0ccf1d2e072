// Weight repack: GPTQ-style int32-packed INT4 codes + bf16 group scales ->
// the tiled layout described in layout.cuh (and its inverse, for round-trip
// checks). Counterpart of the repack step of "The Pivot to Real Hardware ...",
// Step 2 (GPTQ in, hardware-friendly layout out, no act-order permutation);
// the byte count is unchanged.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernels.cuh"

namespace moe {

// Source column (output feature) of tile row r of row tile rt.
//   gate/up GEMM (interleave != 0): row 2i -> gate feature 64*rt + i, row 2i+1 ->
//   up feature N + 64*rt + i, where N = Nout / 2.
//   down GEMM: row r -> feature 128*rt + r.
__device__ __forceinline__ int tile_row_source(int rt, int r, int Nout, int interleave) {
  if (interleave) return rt * 64 + (r >> 1) + (r & 1) * (Nout >> 1);
  return rt * kBM + r;
}

// GPTQ word (code i = element 8*row + i at bits 4i..) -> interleaved word
// (element 2p at bits 4p, element 2p+1 at bits 16 + 4p).
__device__ __forceinline__ uint32_t interleave_codes(uint32_t src) {
  uint32_t dst = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t nib = (src >> (4 * i)) & 0xFu;
    int pos = (i & 1) ? 16 + 4 * (i >> 1) : 4 * (i >> 1);
    dst |= nib << pos;
  }
  return dst;
}
__device__ __forceinline__ uint32_t deinterleave_codes(uint32_t dst) {
  uint32_t src = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    int pos = (i & 1) ? 16 + 4 * (i >> 1) : 4 * (i >> 1);
    src |= ((dst >> pos) & 0xFu) << (4 * i);
  }
  return src;
}

// Scales are kept as fp16 in the packed layout (the tensor-core operand type):
// exact for bf16 scales inside fp16's normal range, which the dequantisation
// needs anyway; the inverse conversion restores the bf16 bits exactly there.
//
// Supported scales: zero, or a finite magnitude in [2^-14, 8160]. Inside that set
// the fp16 scale equals the bf16 one and every dequantised weight (u - 8) * s
// (at most 3 + 8 significant bits, |u - 8| <= 8) is an exact fp16 normal number
// no larger than 65280; outside it a weight would be rounded, flushed or
// infinite, so the repack flags the scale instead.
__device__ __forceinline__ bool scale_supported(uint16_t b) {
  const uint32_t m = b & 0x7FFFu;             // bf16 magnitude bits
  return m == 0 || (m >= 0x3880u && m <= 0x45FFu);  // 0, or 2^-14 .. 8160
}
__device__ __forceinline__ uint16_t bf16_to_f16_bits(uint16_t b) {
  return __half_as_ushort(__float2half_rn(__uint_as_float(static_cast<uint32_t>(b) << 16)));
}
__device__ __forceinline__ uint16_t f16_to_bf16_bits(uint16_t h) {
  const __nv_bfloat16 v = __float2bfloat16_rn(__half2float(__ushort_as_half(h)));
  return *reinterpret_cast<const uint16_t*>(&v);
}

// One CTA per (expert, row tile, k-block) block. `q` is [E, Kred/8, Nout] int32,
// `s` is [E, Kred/32, Nout] bf16; `R` row tiles of 128 rows, `KBn` k-blocks.
__global__ void __launch_bounds__(256) repack_kernel(const uint32_t* __restrict__ q,
                                                     const uint16_t* __restrict__ s,
                                                     uint8_t* __restrict__ out, int Kred,
                                                     int Nout, int R, int KBn, int interleave,
                                                     int32_t* __restrict__ bad_scale) {
  const long long blk = blockIdx.x;
  const int kb = static_cast<int>(blk % KBn);
  const int rt = static_cast<int>((blk / KBn) % R);
  const long long e = blk / (static_cast<long long>(KBn) * R);
  uint8_t* dst = out + blk * kWBlockBytes;
  uint32_t* dw = reinterpret_cast<uint32_t*>(dst);
  uint16_t* ds = reinterpret_cast<uint16_t*>(dst + kWCodeBytes);
  const long long qrows = Kred / 8, srows = Kred / kGroup;
  // codes: thread t -> row r = t % 128 (consecutive threads read neighbouring columns)
  for (int t = threadIdx.x; t < 1024; t += blockDim.x) {
    const int r = t & 127, j = (t >> 7) & 3, h = t >> 9;
    const int f = tile_row_source(rt, r, Nout, interleave);
    const long long row8 = static_cast<long long>(kb) * 8 + h * 4 + j;
    const uint32_t src = q[(e * qrows + row8) * Nout + f];
    dw[h * 512 + r * 4 + j] = interleave_codes(src);
  }
  for (int t = threadIdx.x; t < 256; t += blockDim.x) {
    const int r = t & 127, h = t >> 7;
    const int f = tile_row_source(rt, r, Nout, interleave);
    const uint16_t b = s[(e * srows + kb * 2 + h) * Nout + f];
    if (!scale_supported(b)) *bad_scale = 1;
    ds[r * 2 + h] = bf16_to_f16_bits(b);
  }
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ in,
                                                     uint32_t* __restrict__ q,
                                                     uint16_t* __restrict__ s, int Kred, int Nout,
                                                     int R, int KBn, int interleave) {
  const long long blk = blockIdx.x;
  const int kb = static_cast<int>(blk % KBn);
  const int rt = static_cast<int>((blk / KBn) % R);
  const long long e = blk / (static_cast<long long>(KBn) * R);
  const uint8_t* src = in + blk * kWBlockBytes;
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(src);
  const uint16_t* ss = reinterpret_cast<const uint16_t*>(src + kWCodeBytes);
  const long long qrows = Kred / 8, srows = Kred / kGroup;
  for (int t = threadIdx.x; t < 1024; t += blockDim.x) {
    const int r = t & 127, j = (t >> 7) & 3, h = t >> 9;
    const int f = tile_row_source(rt, r, Nout, interleave);
    const long long row8 = static_cast<long long>(kb) * 8 + h * 4 + j;
    q[(e * qrows + row8) * Nout + f] = deinterleave_codes(sw[h * 512 + r * 4 + j]);
  }
  for (int t = threadIdx.x; t < 256; t += blockDim.x) {
    const int r = t & 127, h = t >> 7;
    const int f = tile_row_source(rt, r, Nout, interleave);
    s[(e * srows + kb * 2 + h) * Nout + f] = f16_to_bf16_bits(ss[r * 2 + h]);
  }
}

cudaError_t launch_repack(const uint32_t* q, const uint16_t* s, uint8_t* out, int E, int Kred,
                          int Nout, int R, int KBn, int interleave, int32_t* bad_scale,
                          cudaStream_t stream) {
  const long long blocks = static_cast<long long>(E) * R * KBn;
  if (blocks <= 0) return cudaSuccess;
  repack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(q, s, out, Kred, Nout, R, KBn,
                                                                   interleave, bad_scale);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* in, uint32_t* q, uint16_t* s, int E, int Kred, int Nout,
                          int R, int KBn, int interleave, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(E) * R * KBn;
  if (blocks <= 0) return cudaSuccess;
  unpack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(in, q, s, Kred, Nout, R, KBn,
                                                                   interleave);
  return cudaGetLastError();
}

}  // namespace moe
