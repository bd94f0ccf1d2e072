// Copying a token row into the B operand: the row's prescale exponent and the
// bf16 -> scaled fp16 conversion (shared by the routing + gather kernels and the
// fused small-batch GEMM, which gathers its rows itself).
#pragma once
#include <cuda_fp16.h>

#include <cstdint>

#include "layout.cuh"

namespace moe {

// Largest magnitude among eight bf16 values, as bf16 magnitude bits: for finite
// values the order of |x| is the order of the low 15 bits.
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  return m;
}

// Prescale exponent of a token row whose largest magnitude has bf16 bits `m`:
// the e for which that magnitude times 2^-e lies in [4, 8) (clamped to
// +-kMaxRowExp); 0 for an all-zero row, and for a row holding an infinity or a
// NaN (outside the supported input range: such values saturate).
__device__ __forceinline__ int row_exponent(uint32_t m) {
  if (m == 0 || m >= 0x7F80u) return 0;
  const int biased = static_cast<int>(m >> 7);
  // floor(log2 |x|): from the exponent field, or for a subnormal (m * 2^-133) from
  // the leading mantissa bit
  const int lg = biased > 0 ? biased - 127 : (31 - __clz(static_cast<int>(m))) - 133;
  const int e = lg - 2;
  return e < -kMaxRowExp ? -kMaxRowExp : (e > kMaxRowExp ? kMaxRowExp : e);
}

// bf16 pair times f -> fp16 pair (f = 2^-e is exact; values stay below 8 for a
// finite row, the clamp only bounds non-finite ones).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float f) {
  const float lo = fminf(fmaxf(__uint_as_float(w << 16) * f, -65504.0f), 65504.0f);
  const float hi = fminf(fmaxf(__uint_as_float(w & 0xFFFF0000u) * f, -65504.0f), 65504.0f);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t bf16_pair(const uint16_t* xr, int a, int b) {
  return static_cast<uint32_t>(__ldg(xr + a)) | (static_cast<uint32_t>(__ldg(xr + b)) << 16);
}

// Blocked B-operand offset of 16-byte chunk ch (8 elements) of padded row p: the
// k-block of 64 elements, the row group of 16 rows, the 128-byte row with its
// 16-byte chunks swizzled by the row (128-byte swizzle of the MMA's B operand).
__device__ __forceinline__ long long b_operand_offset(int ch, int p, int Gcap) {
  const int grp = p / kRowGroup, row = p % kRowGroup;
  return (static_cast<long long>(ch >> 3) * Gcap + grp) * kRowGroupBytes + row * 128 +
         (((ch & 7) ^ (row & 7)) << 4);
}

}  // namespace moe
