// Forward RoPE of the query and of the new KV row, and insertion of the KV
// row into an FP8 (OCP E4M3, per-tensor scale) or BF16 cache (memory-bound).
//
// Page "[ROCm][DSv4] Functional fixes for DeepSeek V4 on MI300X/MI325X",
// Purpose: the fused DeepSeek V4 RoPE / KV-insert path must store the bytes
// of the platform's FP8 encoding (OCP E4M3, maximum 448, on the current
// architecture), with the cache either BF16 or FP8 with one per-tensor scale.
// Layout and rules are stated in include/mxq.h.
//
// Work item = one 16-byte chunk (8 values) of a row outside the rotated
// slice, or one rotate-half pair of chunks inside it (chunk c of the lower
// half and chunk c + R/16, so that both are read before either is written:
// the query may be rotated in place).  Query rows come first, then the KV
// rows; consecutive threads take consecutive chunks of a row, so loads and
// stores are coalesced.  When the query is rotated in place, its chunks
// outside the slice are neither read nor written.  Each rotated value is
// fl32(x0*c -+ x1*s) with both products exact in fp32 (BF16 x BF16), i.e.
// one rounding; the FP8 code is the RNE, saturating E4M3 of the fp32
// quotient fl32(y / scale).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mxq.h"
#include "mxq_internal.h"
#include "quant_common.cuh"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

struct KvArgs {
  const uint4* q;
  uint4* q_out;
  const uint4* kv;
  uint8_t* cache;
  const int64_t* pos;
  const int64_t* slot;
  const uint16_t* cos_tab;
  const uint16_t* sin_tab;
  const float* scale;
  int32_t* err_flag;
  int64_t cs_ld, max_pos, num_slots;
  uint32_t q_items, n_items;  // items of the query rows; of all rows
  uint32_t iq, ik;            // items per query row / per KV row
  uint32_t pq, pk;            // items of a query / KV row outside the slice
  int H, Dq, Dk, R;
  int fp8;                    // 1: E4M3 cache, 0: BF16 cache
};

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint4 to_bf16x8(const float (&y)[8]) {
  return make_uint4(pack2(y[0], y[1]), pack2(y[2], y[3]), pack2(y[4], y[5]), pack2(y[6], y[7]));
}

__device__ __forceinline__ uint2 to_e4m3x8(const float (&y)[8], float scale) {
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = __fdiv_rn(y[e], scale);
  uint2 o;
  o.x = e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16);
  o.y = e4m3x2(v[4], v[5]) | (e4m3x2(v[6], v[7]) << 16);
  return o;
}

// Stores 8 values of KV row chunk c into the cache row `dst` (E4M3 or BF16).
__device__ __forceinline__ void store_cache(const KvArgs& a, uint8_t* dst, int c, const float (&y)[8],
                                            float scale) {
  if (a.fp8)
    *reinterpret_cast<uint2*>(dst + (size_t)c * 8) = to_e4m3x8(y, scale);
  else
    *reinterpret_cast<uint4*>(dst + (size_t)c * 16) = to_bf16x8(y);
}

__global__ void __launch_bounds__(kThreads, kBlocksPerSm) rope_kv_insert_kernel(const KvArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Everything below reads what preceding kernels wrote.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float scale = a.fp8 ? __ldg(a.scale) : 1.0f;
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t it = blockIdx.x * kThreads + threadIdx.x; it < a.n_items; it += stride) {
    const bool is_q = it < a.q_items;
    uint32_t row, i;
    int64_t t;
    if (is_q) {
      row = it / a.iq;
      i = it - row * a.iq;
      t = row / (uint32_t)a.H;
    } else {
      const uint32_t k = it - a.q_items;
      row = k / a.ik;
      i = k - row * a.ik;
      t = row;
    }
    const int D = is_q ? a.Dq : a.Dk;
    const uint32_t plain = is_q ? a.pq : a.pk;
    const uint4* src = (is_q ? a.q : a.kv) + (size_t)row * (D >> 3);
    int64_t p = 0;
    bool bad = false;
    if (a.R > 0) {
      p = __ldg(a.pos + t);
      bad = p < 0 || p >= a.max_pos;
    }
    uint8_t* dst = nullptr;  // this token's cache row (KV items that write)
    if (!is_q) {
      const int64_t sl = __ldg(a.slot + t);
      const bool over = sl >= a.num_slots;
      if (i == 0 && a.err_flag != nullptr && (bad || over))
        atomicOr(a.err_flag, (bad ? MXQ_DEVERR_POSITION : 0) | (over ? MXQ_DEVERR_SLOT : 0));
      if (sl < 0 || over || bad) continue;
      dst = a.cache + (size_t)sl * (size_t)a.Dk * (a.fp8 ? 1 : 2);
    }
    if (i < plain) {
      // A chunk outside the rotated slice: copied (query) or encoded (KV).
      const int c = (int)i;
      const uint4 v = src[c];
      if (is_q) {
        a.q_out[(size_t)row * (D >> 3) + c] = v;
      } else if (a.fp8) {
        float y[8];
        unpack8(v, y);
        store_cache(a, dst, c, y, scale);
      } else {
        *reinterpret_cast<uint4*>(dst + (size_t)c * 16) = v;  // BF16 of a BF16 value: itself
      }
      continue;
    }
    // A rotate-half pair inside the slice: chunks c0 (lower half) and c1.
    const int c0 = (D - a.R) / 8 + (int)(i - plain);
    const int c1 = c0 + a.R / 16;
    float y0[8], y1[8];
    if (bad) {  // invalid position: the query's slice is written as zeros
#pragma unroll
      for (int e = 0; e < 8; ++e) y0[e] = y1[e] = 0.0f;
    } else {
      // Plain loads: the query may be rotated in place (this thread writes
      // these two chunks afterwards; no other thread touches them).
      const uint4 va = src[c0];
      const uint4 vb = src[c1];
      const int j = (int)(i - plain) * 8;  // index into the half (R/2 entries)
      const uint4 cw = __ldg(reinterpret_cast<const uint4*>(a.cos_tab + p * a.cs_ld + j));
      const uint4 sw = __ldg(reinterpret_cast<const uint4*>(a.sin_tab + p * a.cs_ld + j));
      float x0[8], x1[8], c8[8], s8[8];
      unpack8(va, x0);
      unpack8(vb, x1);
      unpack8(cw, c8);
      unpack8(sw, s8);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        y0[e] = __fsub_rn(__fmul_rn(x0[e], c8[e]), __fmul_rn(x1[e], s8[e]));
        y1[e] = __fadd_rn(__fmul_rn(x1[e], c8[e]), __fmul_rn(x0[e], s8[e]));
      }
    }
    if (is_q) {
      uint4* o = a.q_out + (size_t)row * (D >> 3);
      o[c0] = to_bf16x8(y0);
      o[c1] = to_bf16x8(y1);
    } else {
      store_cache(a, dst, c0, y0, scale);
      store_cache(a, dst, c1, y1, scale);
    }
  }
}

}  // namespace

cudaError_t launch_rope_kv_insert(const void* q, void* q_out, int64_t T, int H, int Dq,
                                  const void* kv, int Dk, const int64_t* pos, const void* cos,
                                  const void* sin, int64_t cs_ld, int64_t max_pos, int R,
                                  const int64_t* slot, void* cache, int64_t num_slots, int fp8,
                                  const float* scale, int32_t* err_flag, int num_sms,
                                  cudaStream_t s) {
  KvArgs a = {};
  a.q = reinterpret_cast<const uint4*>(q);
  a.q_out = reinterpret_cast<uint4*>(q_out);
  a.kv = reinterpret_cast<const uint4*>(kv);
  a.cache = static_cast<uint8_t*>(cache);
  a.pos = pos;
  a.slot = slot;
  a.cos_tab = reinterpret_cast<const uint16_t*>(cos);
  a.sin_tab = reinterpret_cast<const uint16_t*>(sin);
  a.scale = scale;
  a.err_flag = err_flag;
  a.cs_ld = cs_ld;
  a.max_pos = max_pos;
  a.num_slots = num_slots;
  a.H = H;
  a.Dq = Dq;
  a.Dk = Dk;
  a.R = R;
  a.fp8 = fp8;
  // In place, the query's chunks outside the slice stay where they are.
  a.pq = (H > 0 && q != q_out) ? (uint32_t)((Dq - R) / 8) : 0u;
  a.pk = (uint32_t)((Dk - R) / 8);
  a.iq = a.pq + (uint32_t)(R / 16);
  a.ik = a.pk + (uint32_t)(R / 16);
  a.q_items = (uint32_t)(T * H) * a.iq;
  a.n_items = a.q_items + (uint32_t)T * a.ik;
  if (a.n_items == 0) return cudaSuccess;
  const int64_t need = ceil_div(a.n_items, kThreads);
  const int64_t cap = (int64_t)num_sms * kBlocksPerSm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(need < cap ? need : cap), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  // Programmatic dependent launch: the grid may be scheduled while the
  // preceding kernel finishes; it waits for it before reading anything.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rope_kv_insert_kernel, a);
}

}  // namespace mxq
