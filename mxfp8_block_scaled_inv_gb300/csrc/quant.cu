// Fused inverse RoPE + group-128 E8M0 / E4M3 quantisation (memory-bound).
//
// Page "[ROCm][DSV4][Perf] Use FP8 WO_A output projection", Summary item 1:
// inverse RoPE on the attention output fused with per-token E8M0 group
// quantisation.  Layout and rules are stated in include/mxq.h.
//
// Mapping: a half-warp (16 lanes) owns one 128-element scale group; each
// lane holds 8 consecutive BF16 values (one 16-byte load).  A warp handles a
// unit of up to 16 consecutive groups of one row: it issues all 8 of its
// 16-byte loads first (two groups per step, one per half-warp), then
// quantises them, so every load instruction of the warp reads 512 contiguous
// bytes and every code store writes 256.  The token's position is read and
// checked once per unit; the RoPE exchange (partner R/16 lanes away in the
// same half-warp) runs only in the step that holds the row's last group.
// The amax is a float abs-max and four xor-shuffles; the exponent comes from
// its bit pattern (no log2, no division).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxq.h"
#include "mxq_internal.h"
#include "quant_common.cuh"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kSteps = 8;  // steps per unit; each step covers two groups
constexpr int kBlocksPerSm = 3;
constexpr int kGroupsPerUnit = 2 * kSteps;

__global__ void __launch_bounds__(kThreads, kBlocksPerSm) inv_rope_group_quant_kernel(
    const uint4* __restrict__ x, uint32_t n_units, int units_per_row, int D, int KG, int R, int G,
    const int64_t* __restrict__ pos, const uint16_t* __restrict__ cos_tab,
    const uint16_t* __restrict__ sin_tab, int64_t cs_ld, int64_t max_pos,
    uint2* __restrict__ q, uint8_t* __restrict__ sc, int32_t* __restrict__ err_flag) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;  // 8-element chunk of the group held by this lane
  const int half = lane >> 4;
  const uint32_t warp = (blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint32_t n_warps = (gridDim.x * kThreads) >> 5;
  const int chunks_per_row = D >> 3;
  // A GEMM launched after this kernel with programmatic dependent launch may
  // start now (it waits for this grid before reading the codes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  for (uint32_t u = warp; u < n_units; u += n_warps) {
    const uint32_t row = u / units_per_row;
    const int g0 = (int)(u - row * units_per_row) * kGroupsPerUnit;
    const size_t rbase = (size_t)row * chunks_per_row;
    int64_t p = 0;
    bool bad = false;
    if (R > 0) {
      p = __ldg(pos + row / G);
      bad = p < 0 || p >= max_pos;
    }
    uint4 v[kSteps];
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
      const int c = (g0 + 2 * s + half) * 16 + sub;
      v[s] = make_uint4(0, 0, 0, 0);
      if (c < chunks_per_row && !bad) v[s] = __ldg(x + rbase + c);
    }
    // Step holding the row's last group (the rotated slice) when R > 0.
    const int rope_step = R > 0 ? ((KG - 1) - g0) >> 1 : -1;
#pragma unroll
    for (int s = 0; s < kSteps; ++s) {
      const int gi = g0 + 2 * s + half;
      if (g0 + 2 * s >= KG) break;  // warp-uniform: nothing left in this unit
      float y[8];
      unpack8(v[s], y);
      if (s == rope_step) {
        // Rotate-half pairs of the last R elements: lanes [16-R/8, 16) of the
        // group's half-warp; partner R/16 lanes away.
        const int first = 16 - (R >> 3);
        const int dist = R >> 4;
        const bool mine = gi == KG - 1 && sub >= first;
        const bool lower = sub < first + dist;
        const int src = (half << 4) | (mine ? (lower ? sub + dist : sub - dist) : sub);
        uint4 pv;
        pv.x = __shfl_sync(0xffffffffu, v[s].x, src);
        pv.y = __shfl_sync(0xffffffffu, v[s].y, src);
        pv.z = __shfl_sync(0xffffffffu, v[s].z, src);
        pv.w = __shfl_sync(0xffffffffu, v[s].w, src);
        if (mine && !bad) {
          const int i0 = (sub - first - (lower ? 0 : dist)) * 8;
          const uint4 cw = __ldg(reinterpret_cast<const uint4*>(cos_tab + p * cs_ld + i0));
          const uint4 sw = __ldg(reinterpret_cast<const uint4*>(sin_tab + p * cs_ld + i0));
          float xp[8];
          unpack8(pv, xp);
          inv_rope8(y, xp, cw, sw, lower);
        }
      }
      const float amax = half_warp_amax(y);
      const int c = gi * 16 + sub;
      if (gi < KG && c < chunks_per_row) {
        uint32_t sbyte;
        uint2 out = encode8(y, amax, &sbyte);
        if (bad) {  // a token with an invalid position is written as zeros
          out = make_uint2(0, 0);
          sbyte = 0;
        }
        q[rbase + c] = out;
        if (sub == 0) sc[(size_t)row * KG + gi] = (uint8_t)sbyte;
      }
    }
    if (bad && lane == 0 && g0 == 0 && err_flag != nullptr) atomicOr(err_flag, MXQ_DEVERR_POSITION);
  }
}

}  // namespace

cudaError_t launch_inv_rope_group_quant(const void* x, int64_t T, int G, int D, int R,
                                        const int64_t* pos, const void* cos, const void* sin,
                                        int64_t cs_ld, int64_t max_pos, uint8_t* q, uint8_t* sc,
                                        int32_t* err_flag, int num_sms, cudaStream_t s) {
  const int KG = (int)ceil_div(D, kGroup);
  const int units_per_row = (int)ceil_div(KG, kGroupsPerUnit);
  const uint32_t n_units = (uint32_t)(T * G * units_per_row);
  const int64_t blocks_needed = ceil_div(n_units, kThreads / 32);
  const int64_t max_blocks = (int64_t)num_sms * kBlocksPerSm;
  const int blocks = (int)(blocks_needed < max_blocks ? blocks_needed : max_blocks);
  inv_rope_group_quant_kernel<<<blocks, kThreads, 0, s>>>(
      reinterpret_cast<const uint4*>(x), n_units, units_per_row, D, KG, R, G, pos,
      reinterpret_cast<const uint16_t*>(cos), reinterpret_cast<const uint16_t*>(sin), cs_ld,
      max_pos, reinterpret_cast<uint2*>(q), sc, err_flag);
  return cudaGetLastError();
}

}  // namespace mxq
