// The 1x128 power-of-two e4m3 activation rule, shared by the input
// quantizer and the GEMM1 epilogue's requantization, and the 1x32 e2m1 rule
// of the FP4-activation variant (UE8M0 exponent per 32 elements, the
// microscaling blocking of the FP4 weights).
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

// n = min{n : amax <= 6 * 2^n} (6 = the largest e2m1 magnitude). With
// amax = m * 2^E, m in [0.5, 1) and 6 = 0.75 * 2^3, n = E - 3 if m <= 0.75
// else E - 2; m <= 0.75 is "fraction bits <= 0x400000". Subnormal amax lands
// below -127 and clamps.
__device__ __forceinline__ int act_exponent_e2m1(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int biased = (b >> 23) & 0xFF;
  if (amax == 0.0f) return 0;
  if (biased == 0) return -127;
  const int E = biased - 126;
  const int n = ((b & 0x7FFFFF) <= 0x400000u) ? E - 3 : E - 2;
  return max(-127, min(127, n));
}

// Eight values to eight e2m1 codes (round to nearest even, saturating),
// packed two per byte with the even element in the low nibble: the
// conversion puts its first operand in the high nibble.
__device__ __forceinline__ uint32_t pack8_e2m1(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                               float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// Word index of (row r, block b) in the scale-word layout.
__device__ __forceinline__ size_t sf_word_index(int r, int b, int nblk) {
  return (static_cast<size_t>(r / 128) * nblk + b) * 128 + 4 * (r % 32) + (r % 128) / 32;
}

}  // namespace bsmoe
