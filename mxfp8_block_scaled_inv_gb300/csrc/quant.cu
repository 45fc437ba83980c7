// Fused inverse RoPE + group-128 E8M0 / E4M3 quantisation (memory-bound).
//
// Page "[ROCm][DSV4][Perf] Use FP8 WO_A output projection", Summary item 1:
// inverse RoPE on the attention output fused with per-token E8M0 group
// quantisation.  Layout and rules are stated in include/mxq.h.
//
// Mapping: a half-warp (16 lanes) owns one 128-element scale group; each
// lane holds 8 consecutive BF16 values (one 16-byte load).  A warp handles
// two adjacent groups per step, so every load instruction of the warp reads
// 512 contiguous bytes and every code store writes 256 contiguous bytes.
// The amax is an xor-shuffle over the 16 lanes; the RoPE partner of an
// element lives R/16 lanes away in the same half-warp.  U steps are issued
// back to back to keep U 16-byte loads in flight per lane.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxq.h"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two OCP E4M3 bytes (round to nearest even, saturating).
// The first source operand of the conversion fills the upper byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kThreads) inv_rope_group_quant_kernel(
    const uint4* __restrict__ x, uint32_t n_groups, int D, int KG, int R, int G,
    const int64_t* __restrict__ pos, const uint16_t* __restrict__ cos_tab,
    const uint16_t* __restrict__ sin_tab, int64_t cs_ld, int64_t max_pos,
    uint2* __restrict__ q, uint8_t* __restrict__ sc, int32_t* __restrict__ err_flag) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;  // lane within the half-warp = 8-element chunk of the group
  const int half = lane >> 4;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t n_warps = (gridDim.x * kThreads) >> 5;
  const int rope_first = (128 - R) >> 3;  // first lane of the rotated slice (R > 0)
  const int rope_dist = R >> 4;           // lane distance between pair partners
  const int chunks_per_row = D >> 3;

  for (uint32_t base = warp * (2 * kUnroll); base < n_groups; base += n_warps * (2 * kUnroll)) {
    uint4 v[kUnroll];
    uint32_t row[kUnroll], kg[kUnroll];
    bool live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t gi = base + 2 * u + half;
      row[u] = gi / KG;
      kg[u] = gi - row[u] * KG;
      live[u] = gi < n_groups && (int)(kg[u] * 16 + sub) < chunks_per_row;
      v[u] = make_uint4(0, 0, 0, 0);
      if (live[u]) v[u] = __ldg(x + (size_t)row[u] * chunks_per_row + kg[u] * 16 + sub);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float y[8] = {bf16_lo(v[u].x), bf16_hi(v[u].x), bf16_lo(v[u].y), bf16_hi(v[u].y),
                    bf16_lo(v[u].z), bf16_hi(v[u].z), bf16_lo(v[u].w), bf16_hi(v[u].w)};
      bool bad = false;
      if (R > 0) {
        // Every group of a token with an invalid position is zeroed.
        const bool in_range = base + 2 * u + half < n_groups;
        const int64_t p = in_range ? __ldg(pos + row[u] / G) : 0;
        bad = in_range && (p < 0 || p >= max_pos);
        const bool rope_group = in_range && (int)kg[u] == KG - 1;
        const bool mine = rope_group && sub >= rope_first;
        const bool lower = sub < rope_first + rope_dist;
        const int partner = mine ? (lower ? sub + rope_dist : sub - rope_dist) : sub;
        const int src = (half << 4) | partner;
        uint4 pv;
        pv.x = __shfl_sync(0xffffffffu, v[u].x, src);
        pv.y = __shfl_sync(0xffffffffu, v[u].y, src);
        pv.z = __shfl_sync(0xffffffffu, v[u].z, src);
        pv.w = __shfl_sync(0xffffffffu, v[u].w, src);
        if (mine && !bad) {
          const int i0 = (sub - rope_first - (lower ? 0 : rope_dist)) * 8;
          const uint4 cw = __ldg(reinterpret_cast<const uint4*>(cos_tab + p * cs_ld + i0));
          const uint4 sw = __ldg(reinterpret_cast<const uint4*>(sin_tab + p * cs_ld + i0));
          const float c[8] = {bf16_lo(cw.x), bf16_hi(cw.x), bf16_lo(cw.y), bf16_hi(cw.y),
                              bf16_lo(cw.z), bf16_hi(cw.z), bf16_lo(cw.w), bf16_hi(cw.w)};
          const float s[8] = {bf16_lo(sw.x), bf16_hi(sw.x), bf16_lo(sw.y), bf16_hi(sw.y),
                              bf16_lo(sw.z), bf16_hi(sw.z), bf16_lo(sw.w), bf16_hi(sw.w)};
          const float xp[8] = {bf16_lo(pv.x), bf16_hi(pv.x), bf16_lo(pv.y), bf16_hi(pv.y),
                               bf16_lo(pv.z), bf16_hi(pv.z), bf16_lo(pv.w), bf16_hi(pv.w)};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // lower half: y0 = x0*c + x1*s ; upper half: y1 = x1*c - x0*s.
            // Products of two BF16 values are exact in fp32; one rounding each.
            y[e] = lower ? __fadd_rn(__fmul_rn(y[e], c[e]), __fmul_rn(xp[e], s[e]))
                         : __fsub_rn(__fmul_rn(y[e], c[e]), __fmul_rn(xp[e], s[e]));
          }
        }
      }
      // Group amax as the largest magnitude bit pattern (non-negative floats
      // order like unsigned integers).
      uint32_t m = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = max(m, __float_as_uint(y[e]) & 0x7FFFFFFFu);
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      if (!live[u]) continue;
      // Smallest e with amax <= 448 * 2^e.  amax = (1+f) * 2^E with
      // 448 = 1.75 * 2^8: e = E - 8 + (f > 0.75); zero/subnormal amax and
      // anything below 2^-127 * 448 clamp to e = -127.
      const int bexp = (int)(m >> 23);
      int ex = bexp - 127 - 8 + ((m & 0x7FFFFFu) > 0x600000u ? 1 : 0);
      ex = bexp == 0 ? -127 : max(ex, -127);
      uint32_t sbyte = (uint32_t)(ex + 127);
      float inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-e, -e in [-120, 127]
      if (bexp == 255) {  // non-finite input: outside the contract
        sbyte = 0xFF;
        inv = 1.0f;
      }
      uint2 out;
      out.x = e4m3x2(__fmul_rn(y[0], inv), __fmul_rn(y[1], inv)) |
              (e4m3x2(__fmul_rn(y[2], inv), __fmul_rn(y[3], inv)) << 16);
      out.y = e4m3x2(__fmul_rn(y[4], inv), __fmul_rn(y[5], inv)) |
              (e4m3x2(__fmul_rn(y[6], inv), __fmul_rn(y[7], inv)) << 16);
      if (bad) {
        out = make_uint2(0, 0);
        sbyte = 0;
      }
      q[((size_t)row[u] * chunks_per_row + kg[u] * 16 + sub)] = out;
      if (sub == 0) {
        sc[(size_t)row[u] * KG + kg[u]] = (uint8_t)sbyte;
        if (bad && err_flag != nullptr) atomicOr(err_flag, MXQ_DEVERR_POSITION);
      }
    }
  }
}

}  // namespace

cudaError_t launch_inv_rope_group_quant(const void* x, int64_t T, int G, int D, int R,
                                        const int64_t* pos, const void* cos, const void* sin,
                                        int64_t cs_ld, int64_t max_pos, uint8_t* q, uint8_t* sc,
                                        int32_t* err_flag, int num_sms, cudaStream_t s) {
  const int KG = (int)ceil_div(D, kGroup);
  const uint32_t n_groups = (uint32_t)(T * G * KG);
  const int64_t warps_needed = ceil_div(n_groups, 2 * kUnroll);
  const int64_t blocks_needed = ceil_div(warps_needed, kThreads / 32);
  const int64_t max_blocks = (int64_t)num_sms * (2048 / kThreads);
  const int blocks = (int)(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  inv_rope_group_quant_kernel<<<blocks, kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(x), n_groups, D, KG, R, G, pos,
      reinterpret_cast<const uint16_t*>(cos), reinterpret_cast<const uint16_t*>(sin), cs_ld,
      max_pos, reinterpret_cast<uint2*>(q), sc, err_flag);
  return cudaGetLastError();
}

}  // namespace mxq
