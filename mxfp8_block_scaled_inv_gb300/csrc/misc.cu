// Load-time kernels: MXFP8 -> BF16 dequantisation, the weight-scale layout
// transform the block-scaled GEMM reads, and FP32 power-of-two scales ->
// E8M0 bytes.  Contracts are stated in include/mxq.h.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "mxq.h"
#include "mxq_internal.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;

// Two E4M3 bytes (low byte first) -> two fp32 values, exactly (every E4M3
// value is an fp16 value).
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// 2^(byte-127) as fp32: byte 0 is the subnormal 2^-127, 0xFF is NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 0) return __uint_as_float(0x00400000u);
  if (b == 255) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(b << 23);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);  // round to nearest even, each half
  return *reinterpret_cast<uint32_t*>(&r);
}

// Dequantisation-once page, Purpose: out = bf16(E4M3(code) * 2^(scale-127)).
// One thread per 16 codes: a 16-byte load, two 16-byte stores.  The product
// is exact in fp32 (4 significant bits times a power of two, above 2^-149)
// or overflows fp32 exactly when the BF16 result overflows too, so the only
// rounding is the final fp32 -> BF16.
__global__ void __launch_bounds__(kThreads) dequant_bf16_kernel(
    const uint4* __restrict__ w, const uint8_t* __restrict__ sc, uint4* __restrict__ out,
    uint32_t n_chunks, uint32_t chunks_per_row, int KG) {
  // Launched with programmatic dependent launch: wait for the preceding
  // kernel's writes before reading, and let the next kernel start launching.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (uint32_t c = blockIdx.x * kThreads + threadIdx.x; c < n_chunks; c += gridDim.x * kThreads) {
    const uint32_t row = c / chunks_per_row;
    const uint32_t kc = c - row * chunks_per_row;
    const float scale = e8m0_to_f32(__ldg(sc + (size_t)row * KG + (kc >> 3)));
    const uint4 v = __ldg(w + c);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = e4m3x2_to_f32((uint16_t)(words[i] & 0xFFFF));
      const float2 b = e4m3x2_to_f32((uint16_t)(words[i] >> 16));
      o[2 * i] = pack_bf16x2(__fmul_rn(a.x, scale), __fmul_rn(a.y, scale));
      o[2 * i + 1] = pack_bf16x2(__fmul_rn(b.x, scale), __fmul_rn(b.y, scale));
    }
    out[2 * (size_t)c] = make_uint4(o[0], o[1], o[2], o[3]);
    out[2 * (size_t)c + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// Prepared weight-scale layout: for each (b, kg, 128-row block nb) a
// 512-byte atom; row r = 32*j + i of the block owns the word at byte
// 16*i + 4*j, holding its scale byte four times.  Rows past N hold 127.
__global__ void __launch_bounds__(kThreads) prepare_weight_scales_kernel(
    const uint8_t* __restrict__ in, uint32_t* __restrict__ out, uint32_t n_words, int N, int KG,
    int NB) {
  for (uint32_t w = blockIdx.x * kThreads + threadIdx.x; w < n_words; w += gridDim.x * kThreads) {
    const uint32_t atom = w >> 7;
    const uint32_t within = w & 127;
    const uint32_t i = within >> 2, j = within & 3;
    const uint32_t nb = atom % NB;
    const uint32_t bk = atom / NB;  // b * KG + kg
    const uint32_t kg = bk % KG;
    const uint32_t b = bk / KG;
    const uint32_t r = nb * 128 + 32 * j + i;
    const uint32_t byte = r < (uint32_t)N ? in[((size_t)b * N + r) * KG + kg] : 127u;
    out[w] = byte * 0x01010101u;
  }
}

// FP8 WO_A page, Implementation: an FP32 scale that is an exact power of two
// maps to its biased exponent; the bits are inspected, no FP8 arithmetic.
__global__ void __launch_bounds__(kThreads) scales_f32_to_e8m0_kernel(
    const uint32_t* __restrict__ s, uint8_t* __restrict__ out, int64_t n,
    int32_t* __restrict__ err_flag) {
  for (int64_t i = blockIdx.x * (int64_t)kThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kThreads) {
    const uint32_t b = __ldg(s + i);
    const uint32_t bexp = b >> 23;  // includes the sign bit: negative values fail below
    const uint32_t man = b & 0x7FFFFFu;
    uint32_t byte = 0xFF;
    if (bexp >= 1 && bexp <= 254 && man == 0) byte = bexp;  // 2^(bexp-127), k in [-126, 127]
    else if (b == 0x00400000u) byte = 0;                    // 2^-127 (subnormal)
    out[i] = (uint8_t)byte;
    if (byte == 0xFF && err_flag != nullptr) atomicOr(err_flag, MXQ_DEVERR_SCALE);
  }
}

int grid_for(int64_t work, int per_block, int num_sms) {
  const int64_t need = ceil_div(work, per_block);
  const int64_t cap = (int64_t)num_sms * (2048 / kThreads) * 4;
  return (int)(need < cap ? (need < 1 ? 1 : need) : cap);
}

}  // namespace

cudaError_t launch_dequant_bf16(const uint8_t* w, const uint8_t* sc, void* out, int B, int N, int K,
                                int num_sms, cudaStream_t s) {
  const uint32_t chunks_per_row = (uint32_t)(K / 16);
  const uint32_t n_chunks = (uint32_t)((int64_t)B * N * chunks_per_row);
  const int KG = (int)ceil_div(K, kGroup);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_for(n_chunks, kThreads, num_sms), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dequant_bf16_kernel, reinterpret_cast<const uint4*>(w), sc,
                            reinterpret_cast<uint4*>(out), n_chunks, chunks_per_row, KG);
}

cudaError_t launch_prepare_weight_scales(const uint8_t* w_e8m0, int B, int N, int K, uint8_t* out,
                                         cudaStream_t s) {
  const int KG = (int)ceil_div(K, kGroup);
  const int NB = (int)sf_row_blocks(N);
  const uint32_t n_words = (uint32_t)((int64_t)B * KG * NB * (kSfAtomBytes / 4));
  prepare_weight_scales_kernel<<<grid_for(n_words, kThreads, 148), kThreads, 0, s>>>(
      w_e8m0, reinterpret_cast<uint32_t*>(out), n_words, N, KG, NB);
  return cudaGetLastError();
}

cudaError_t launch_scales_f32_to_e8m0(const float* s, int64_t n, uint8_t* out, int32_t* err_flag,
                                      cudaStream_t st) {
  scales_f32_to_e8m0_kernel<<<grid_for(n, kThreads, 148), kThreads, 0, st>>>(
      reinterpret_cast<const uint32_t*>(s), out, n, err_flag);
  return cudaGetLastError();
}

}  // namespace mxq
