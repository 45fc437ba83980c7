// Per-group quantisation arithmetic shared by the standalone quantiser and
// the GEMM's fused activation path: one half-warp holds one 128-element
// group, each lane 8 consecutive values.
//
// Page "[ROCm][DSV4][Perf] Use FP8 WO_A output projection", Summary item 1
// (per-token E8M0 group quantisation); page "[ROCm][DSv4] Functional fixes
// for DeepSeek V4 on MI300X/MI325X", Purpose (OCP E4M3, maximum 448).
#pragma once

#include <stdint.h>

namespace mxq {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two OCP E4M3 bytes (round to nearest even, saturating).
// The first source operand of the conversion fills the upper byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantises one lane's 8 values of a group whose amax (over the 16 lanes of
// the half-warp) is `amax`; returns the 8 codes and the group's scale byte.
__device__ __forceinline__ uint2 encode8(const float (&y)[8], float amax, uint32_t* sbyte) {
  // Smallest e with amax <= 448 * 2^e: amax = (1+f) * 2^E and 448 = 1.75 * 2^8
  // give e = E - 8 + (f > 0.75); zero / subnormal amax clamps to e = -127.
  const uint32_t m = __float_as_uint(amax);
  const int bexp = (int)(m >> 23);
  int ex = bexp - 127 - 8 + ((m & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  ex = bexp == 0 ? -127 : max(ex, -127);
  float inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-e, -e in [-120, 127]
  *sbyte = (uint32_t)(ex + 127);
  if (bexp == 255) {  // non-finite input: outside the contract
    *sbyte = 0xFF;
    inv = 1.0f;
  }
  uint2 out;
  out.x = e4m3x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) |
          (e4m3x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 16);
  out.y = e4m3x2(__fmul_rn(y[4], inv), __fmul_rn(y[5], inv)) |
          (e4m3x2(__fmul_rn(y[6], inv), __fmul_rn(y[7], inv)) << 16);
  return out;
}

__device__ __forceinline__ float half_warp_amax(const float (&y)[8]) {
  float m = fmaxf(fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3]))),
                  fmaxf(fmaxf(fabsf(y[4]), fabsf(y[5])), fmaxf(fabsf(y[6]), fabsf(y[7]))));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  return m;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&y)[8]) {
  y[0] = bf16_lo(v.x);
  y[1] = bf16_hi(v.x);
  y[2] = bf16_lo(v.y);
  y[3] = bf16_hi(v.y);
  y[4] = bf16_lo(v.z);
  y[5] = bf16_hi(v.z);
  y[6] = bf16_lo(v.w);
  y[7] = bf16_hi(v.w);
}


// Inverse rotation of one lane's 8 values against its partner lane's 8
// values (rotate-half pair, partner R/16 lanes away): the lower half of the
// slice takes y0 = x0*c + x1*s, the upper half y1 = x1*c - x0*s.  Products
// of two BF16 values are exact in fp32, so each output is one rounding.
__device__ __forceinline__ void inv_rope8(float (&y)[8], const float (&xp)[8], const uint4& cw,
                                          const uint4& sw, bool lower) {
  float c8[8], s8[8];
  unpack8(cw, c8);
  unpack8(sw, s8);
#pragma unroll
  for (int e = 0; e < 8; ++e)
    y[e] = lower ? __fadd_rn(__fmul_rn(y[e], c8[e]), __fmul_rn(xp[e], s8[e]))
                 : __fsub_rn(__fmul_rn(y[e], c8[e]), __fmul_rn(xp[e], s8[e]));
}

}  // namespace mxq
