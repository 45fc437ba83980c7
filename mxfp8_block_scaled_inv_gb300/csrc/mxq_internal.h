// Internal declarations shared by the C-ABI layer (api.cpp) and the kernel
// translation units.  Launchers assume their arguments were validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mxq {

constexpr int kGroup = 128;        // scale-group width along the contraction axis
constexpr int kSfAtomBytes = 512;  // one 128-row x 4-byte scale-factor atom
constexpr int kSfRowPad = 256;     // prepared weight-scale rows are padded to this

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of 128-row atoms per (b, kg) in the prepared weight-scale layout.
inline int64_t sf_row_blocks(int64_t N) { return ceil_div(N, kSfRowPad) * (kSfRowPad / 128); }

cudaError_t launch_inv_rope_group_quant(const void* x, int64_t T, int G, int D, int R,
                                        const int64_t* pos, const void* cos, const void* sin,
                                        int64_t cs_ld, int64_t max_pos, uint8_t* q, uint8_t* sc,
                                        int32_t* err_flag, int num_sms, cudaStream_t s);

cudaError_t launch_prepare_weight_scales(const uint8_t* w_e8m0, int B, int N, int K, uint8_t* out,
                                         cudaStream_t s);

cudaError_t launch_dequant_bf16(const uint8_t* w, const uint8_t* sc, void* out, int B, int N, int K,
                                int num_sms, cudaStream_t s);

cudaError_t launch_scales_f32_to_e8m0(const float* s, int64_t n, uint8_t* out, int32_t* err_flag,
                                      cudaStream_t st);

// Block-scaled GEMM.  Returns cudaSuccess or the first CUDA error; a
// non-CUDA failure (e.g. tensor-map encoding) is reported as
// cudaErrorInvalidValue with detail text in *why.
cudaError_t launch_bmm_a8w8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* w,
                            const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                            int num_sms, cudaStream_t s, const char** why);

// One-launch wo_a / MXFP8 linear for T <= 32 tokens: the GEMM reads the BF16
// activation and quantises it itself (inverse RoPE when R > 0).  Above 32
// tokens the per-stage quantisation inside the GEMM costs more than a
// separate quantiser launch, so those calls use two kernels.
constexpr int kFusedMaxTokens = 32;
cudaError_t launch_wo_a_fused(const void* x, const int64_t* pos, const void* cos, const void* sin,
                              int64_t cs_ld, int64_t max_pos, int R, const uint8_t* w,
                              const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                              int32_t* err_flag, int num_sms, cudaStream_t s, const char** why);

// One-launch wo_a for T > 128 tokens: the CTA-pair GEMM with quantising
// warps (inverse RoPE when R > 0) that fill the workspace `ws` (layout
// below, woa_prefill_layout(T, G, K).total bytes, 256-byte aligned).
constexpr int kPairMinTokens = 129;
cudaError_t launch_wo_a_prefill(const void* x, const int64_t* pos, const void* cos, const void* sin,
                                int64_t cs_ld, int64_t max_pos, int R, const uint8_t* w,
                                const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                                int32_t* err_flag, void* ws, int num_sms, cudaStream_t s,
                                const char** why);

// Workspace of launch_wo_a_prefill, each region 256-byte aligned: E4M3 codes
// [T][G][K]; activation scale atoms [G][MB][KG][512] with MB = 2*ceil(T/256)
// 128-token blocks and KG = ceil(K/128); job counters [G][MB][KG] uint32.
struct WoaPrefillLayout {
  size_t codes, atoms, flags, total;
};
inline size_t round_up_256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
inline WoaPrefillLayout woa_prefill_layout(int64_t T, int G, int K) {
  const size_t MB = 2 * (size_t)ceil_div(T, 256);
  const size_t jobs = (size_t)G * MB * (size_t)ceil_div(K, kGroup);
  WoaPrefillLayout l;
  l.codes = 0;
  l.atoms = round_up_256((size_t)T * G * K);
  l.flags = l.atoms + round_up_256(jobs * kSfAtomBytes);
  l.total = l.flags + round_up_256(jobs * 4);
  return l;
}

// Forward RoPE of q [T][H][Dq] into q_out (may equal q) and of kv [T][Dk],
// whose rows go to cache rows slot[t] (E4M3 of fl32(y / *scale) when fp8,
// else BF16).
cudaError_t launch_rope_kv_insert(const void* q, void* q_out, int64_t T, int H, int Dq,
                                  const void* kv, int Dk, const int64_t* pos, const void* cos,
                                  const void* sin, int64_t cs_ld, int64_t max_pos, int R,
                                  const int64_t* slot, void* cache, int64_t num_slots, int fp8,
                                  const float* scale, int32_t* err_flag, int num_sms,
                                  cudaStream_t s);

// Caps the CTA pairs of the pair-form GEMM launches (0 = no cap); returns
// the previous cap.
int set_pair_limit(int pairs);
// Pairs of the quantising form from this index on skip their quantisation
// jobs (a negative value: none); returns the previous setting.
int set_lazy_pairs(int from);

cudaError_t watchdog_read(uint32_t* value, bool clear);
// Device address of the watchdog word on the current device (for kernels of
// other translation units).
cudaError_t watchdog_address(uint32_t** p);
// Number of prefill quantisation jobs taken over by a consumer since the
// last clear (current device).
cudaError_t takeover_count(uint32_t* value, bool clear);

// One tiny kernel whose only wait can never be satisfied; it must give up
// after limit_ns and set bit 31 of the watchdog word.
cudaError_t launch_watchdog_selftest(uint64_t limit_ns, cudaStream_t s);

// Stores `text` as the calling thread's last-error text (mxq_last_error) and
// returns `status`.
int set_error(int status, const char* text);

}  // namespace mxq
