// Weight repack: int32-packed INT4 codes + bf16 group scales (GPTQ or
// compressed-tensors layout, optionally quantised in activation order) -> the
// tiled layout described in layout.cuh (and its inverse, for round-trip checks).
// Counterpart of the repack step of "The Pivot to Real Hardware ...", Step 2
// (GPTQ in, with an act-order permutation or without, hardware-friendly layout
// out); the byte count is unchanged.
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

// Bit position of code i (element 8*row + i of a GPTQ word) in a packed word:
// the codes of pair p = i / 2 (fp16 pair p of the A operand) sit where the
// dequantisation finds them at bits 6..9 (low half) and 22..25 (high half) of
// the word itself (p = 0), shifted left by 4 (p = 1), shifted right by 4 (p = 2)
// or rotated left by 8 (p = 3: bits 30, 31, 0, 1 and 14..17).
__device__ __forceinline__ int code_pos(int i) {
  const int p = i >> 1, h = i & 1;
  return p == 0 ? (h ? 22 : 6) : p == 1 ? (h ? 18 : 2) : p == 2 ? (h ? 26 : 10) : (h ? 14 : 30);
}
// GPTQ word (code i at bits 4i..4i+3) -> packed word, and back.
__device__ __forceinline__ uint32_t interleave_codes(uint32_t src) {
  uint32_t dst = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t nib = (src >> (4 * i)) & 0xFu;
    dst |= __funnelshift_l(nib, nib, code_pos(i));  // a rotation: code 6 wraps past bit 31
  }
  return dst;
}
__device__ __forceinline__ uint32_t deinterleave_codes(uint32_t dst) {
  uint32_t src = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) src |= (__funnelshift_r(dst, dst, code_pos(i)) & 0xFu) << (4 * i);
  return src;
}

// Scales are kept as fp16 in the packed layout (the tensor-core operand type):
// exact for bf16 scales inside fp16's normal range, which the dequantisation
// needs anyway; the inverse conversion restores the bf16 bits exactly there.
//
// Supported scales: zero, or a finite magnitude in [2^-14, 2720]. Inside that set
// the fp16 scale equals the bf16 one, -24 s (the dequantisation's offset term) is
// an exact fp16 number, and every dequantised weight (u - 8) * s (at most 3 + 8
// significant bits, |u - 8| <= 8) is an exact fp16 normal number no larger than
// 21760; outside it a weight would be rounded, flushed or infinite, so the repack
// flags the scale instead.
__device__ __forceinline__ bool scale_supported(uint16_t b) {
  const uint32_t m = b & 0x7FFFu;             // bf16 magnitude bits
  return m == 0 || (m >= 0x3880u && m <= 0x452Au);  // 0, or 2^-14 .. 2720
}
__device__ __forceinline__ uint16_t bf16_to_f16_bits(uint16_t b) {
  return __half_as_ushort(__float2half_rn(__uint_as_float(static_cast<uint32_t>(b) << 16)));
}
__device__ __forceinline__ uint16_t f16_to_bf16_bits(uint16_t h) {
  const __nv_bfloat16 v = __float2bfloat16_rn(__half2float(__ushort_as_half(h)));
  return *reinterpret_cast<const uint16_t*>(&v);
}

// Where a packed element comes from. The codes and scales arrive in one of two
// layouts (`layout`):
//   kLayoutGptq: q [E, Kred/8, Nout] int32, s [E, Kred/32, Nout] -- eight codes of
//     one output feature along the reduction axis per word;
//   kLayoutCompressedTensors: q [E, Nout, Kred/8], s [E, Nout, Kred/32] -- every
//     output feature's row contiguous, the same eight-codes-per-word order.
// With act-order the packed reduction element j of expert e is source element
// red_perm[e][j] (the elements sorted by scale group, so that packed group j/32 is
// source group j/32), and an output-feature permutation (out_perm, period P:
// feature f -> P * (f / P) + out_perm[e][f % P]) may reorder the features.
struct PackSrc {
  const uint32_t* q;
  const uint16_t* s;
  int layout;
  const int32_t* red_perm;  // [E, Kred] or null
  const int32_t* out_perm;  // [E, P] or null
  int out_period;
  int Kred, Nout;
};

__device__ __forceinline__ long long q_index(const PackSrc& p, long long e, int r8, int f) {
  return p.layout == kLayoutGptq ? (e * (p.Kred / 8) + r8) * p.Nout + f
                                 : (e * p.Nout + f) * (p.Kred / 8) + r8;
}
__device__ __forceinline__ long long s_index(const PackSrc& p, long long e, int g, int f) {
  return p.layout == kLayoutGptq ? (e * (p.Kred / kGroup) + g) * p.Nout + f
                                 : (e * p.Nout + f) * (p.Kred / kGroup) + g;
}
__device__ __forceinline__ int source_feature(const PackSrc& p, long long e, int f) {
  if (!p.out_perm) return f;
  const int P = p.out_period;
  return (f / P) * P + p.out_perm[e * P + f % P];
}

// Codes of packed reduction elements 8*r8 .. 8*r8+7 of source feature f (GPTQ
// word order: element 8*r8+i in bits 4i..).
__device__ __forceinline__ uint32_t gather_word(const PackSrc& p, long long e, int r8, int f) {
  if (!p.red_perm) return p.q[q_index(p, e, r8, f)];
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int k = p.red_perm[e * p.Kred + 8 * r8 + i];
    w |= ((p.q[q_index(p, e, k >> 3, f)] >> (4 * (k & 7))) & 0xFu) << (4 * i);
  }
  return w;
}

// One CTA per (expert, row tile, k-block) block; `R` row tiles of 128 rows,
// `KBn` k-blocks of 64 reduction elements.
__global__ void __launch_bounds__(256) repack_kernel(const PackSrc p, uint8_t* __restrict__ out,
                                                     int R, int KBn, int interleave,
                                                     int32_t* __restrict__ bad_scale) {
  const long long blk = blockIdx.x;
  const int kb = static_cast<int>(blk % KBn);
  const int rt = static_cast<int>((blk / KBn) % R);
  const long long e = blk / (static_cast<long long>(KBn) * R);
  uint8_t* dst = out + blk * kWBlockBytes;
  uint32_t* dw = reinterpret_cast<uint32_t*>(dst);
  uint16_t* ds = reinterpret_cast<uint16_t*>(dst + kWCodeBytes);
  // codes: thread t -> row r = t % 128 (consecutive threads read neighbouring columns)
  for (int t = threadIdx.x; t < 1024; t += blockDim.x) {
    const int r = t & 127, j = (t >> 7) & 3, h = t >> 9;
    const int f = source_feature(p, e, tile_row_source(rt, r, p.Nout, interleave));
    dw[h * 512 + r * 4 + j] = interleave_codes(gather_word(p, e, kb * 8 + h * 4 + j, f));
  }
  // scales: packed group kb*2 + h is source group kb*2 + h (act-order sorts the
  // elements by group)
  for (int t = threadIdx.x; t < 256; t += blockDim.x) {
    const int r = t & 127, h = t >> 7;
    const int f = source_feature(p, e, tile_row_source(rt, r, p.Nout, interleave));
    const uint16_t b = p.s[s_index(p, e, kb * 2 + h, f)];
    if (!scale_supported(b)) *bad_scale = 1;
    ds[r * 2 + h] = bf16_to_f16_bits(b);
  }
}

// Inverse of repack_kernel into the source layout (q must be zeroed first when a
// reduction permutation scatters single codes: they are OR-ed into place).
__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ in, PackSrc p,
                                                     uint32_t* __restrict__ q, uint16_t* __restrict__ s,
                                                     int R, int KBn, int interleave) {
  const long long blk = blockIdx.x;
  const int kb = static_cast<int>(blk % KBn);
  const int rt = static_cast<int>((blk / KBn) % R);
  const long long e = blk / (static_cast<long long>(KBn) * R);
  const uint8_t* src = in + blk * kWBlockBytes;
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(src);
  const uint16_t* ss = reinterpret_cast<const uint16_t*>(src + kWCodeBytes);
  for (int t = threadIdx.x; t < 1024; t += blockDim.x) {
    const int r = t & 127, j = (t >> 7) & 3, h = t >> 9;
    const int f = source_feature(p, e, tile_row_source(rt, r, p.Nout, interleave));
    const int r8 = kb * 8 + h * 4 + j;
    const uint32_t w = deinterleave_codes(sw[h * 512 + r * 4 + j]);
    if (!p.red_perm) {
      q[q_index(p, e, r8, f)] = w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = p.red_perm[e * p.Kred + 8 * r8 + i];
        atomicOr(q + q_index(p, e, k >> 3, f), ((w >> (4 * i)) & 0xFu) << (4 * (k & 7)));
      }
    }
  }
  for (int t = threadIdx.x; t < 256; t += blockDim.x) {
    const int r = t & 127, h = t >> 7;
    const int f = source_feature(p, e, tile_row_source(rt, r, p.Nout, interleave));
    s[s_index(p, e, kb * 2 + h, f)] = f16_to_bf16_bits(ss[r * 2 + h]);
  }
}

// Act-order: the packing order of each expert's reduction elements from its group
// index g_idx [E, R] -- the elements of group 0 in ascending index, then those of
// group 1, ... (a stable sort by group). Every group must hold exactly 32
// elements (the layout keeps one scale per 32 consecutive packed elements); an
// index outside [0, R/32) or a group of another size sets *bad. One warp per
// expert; the running count of every group lives in shared memory.
__global__ void __launch_bounds__(32) perm_from_g_idx_kernel(const int32_t* __restrict__ g_idx,
                                                             int32_t* __restrict__ perm, int R,
                                                             int32_t* __restrict__ bad) {
  extern __shared__ int cnt[];
  const int G = R / kGroup;
  const long long e = blockIdx.x;
  const int lane = threadIdx.x;
  for (int i = lane; i < G; i += 32) cnt[i] = 0;
  __syncwarp();
  for (int base = 0; base < R; base += 32) {
    const int k = base + lane;  // R is a multiple of 32
    const int g = g_idx[e * R + k];
    const bool ok = g >= 0 && g < G;
    if (!ok) *bad = 1;
    // lanes of the same group, in lane (= element) order; a bad lane stands alone
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? g : -1 - lane);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int c = ok ? cnt[g] : 0;
    __syncwarp();
    if (ok && rank == 0) cnt[g] = c + __popc(peers);
    __syncwarp();
    if (ok) {
      const int pos = c + rank;
      if (pos < kGroup)
        perm[e * R + g * kGroup + pos] = k;
      else
        *bad = 1;
    }
  }
}

cudaError_t launch_repack(const RepackSource& src, uint8_t* out, int E, int R, int KBn,
                          int interleave, int32_t* bad_scale, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(E) * R * KBn;
  if (blocks <= 0) return cudaSuccess;
  const PackSrc p{reinterpret_cast<const uint32_t*>(src.q), src.s, src.layout, src.red_perm,
                  src.out_perm, src.out_period, src.Kred, src.Nout};
  repack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p, out, R, KBn, interleave,
                                                                   bad_scale);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* in, const RepackSource& dst, int32_t* q, uint16_t* s, int E,
                          int R, int KBn, int interleave, cudaStream_t stream) {
  const long long blocks = static_cast<long long>(E) * R * KBn;
  if (blocks <= 0) return cudaSuccess;
  if (dst.red_perm) {
    cudaError_t e = cudaMemsetAsync(q, 0, static_cast<size_t>(E) * dst.Kred / 8 * dst.Nout * 4, stream);
    if (e != cudaSuccess) return e;
  }
  const PackSrc p{nullptr, nullptr, dst.layout, dst.red_perm, dst.out_perm, dst.out_period,
                  dst.Kred, dst.Nout};
  unpack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      in, p, reinterpret_cast<uint32_t*>(q), s, R, KBn, interleave);
  return cudaGetLastError();
}

cudaError_t launch_perm_from_g_idx(const int32_t* g_idx, int32_t* perm, int E, int R, int32_t* bad,
                                   cudaStream_t stream) {
  if (E <= 0) return cudaSuccess;
  perm_from_g_idx_kernel<<<E, 32, (R / kGroup) * sizeof(int), stream>>>(g_idx, perm, R, bad);
  return cudaGetLastError();
}

}  // namespace moe
