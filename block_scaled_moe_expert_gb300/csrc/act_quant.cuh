// The 1x128 power-of-two e4m3 activation rule, shared by the input
// quantizer and the GEMM1 epilogue's requantization.
#pragma once
#include <cstdint>
#include <cuda_fp8.h>

namespace bsmoe {

// e = min{n : amax <= 448 * 2^n}. With amax = m * 2^E, m in [0.5, 1) and
// 448 = 0.875 * 2^9, n = E - 9 if m <= 0.875 else E - 8; m <= 0.875 is
// "fraction bits <= 0x600000". Subnormal amax lands below -127 and clamps.
__device__ __forceinline__ int act_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int biased = (b >> 23) & 0xFF;
  if (amax == 0.0f) return 0;
  if (biased == 0) return -127;
  const int E = biased - 126;
  const int n = ((b & 0x7FFFFF) <= 0x600000u) ? E - 9 : E - 8;
  return max(-127, min(127, n));
}

// 2^-e as a float for e in [-127, 127] (2^-127 is the one subnormal case).
__device__ __forceinline__ float exp2_neg(int e) {
  return (e == 127) ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Word index of (row r, block b) in the scale-word layout.
__device__ __forceinline__ size_t sf_word_index(int r, int b, int nblk) {
  return (static_cast<size_t>(r / 128) * nblk + b) * 128 + 4 * (r % 32) + (r % 128) / 32;
}

}  // namespace bsmoe
