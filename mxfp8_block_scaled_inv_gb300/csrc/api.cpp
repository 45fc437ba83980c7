// C ABI of libmxq: argument validation, device checks and dispatch to the
// kernel launchers.  Every argument check runs on the host before anything
// is enqueued, so an invalid call launches nothing.  Contracts are in
// include/mxq.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int ok() {
  g_last_error[0] = '\0';
  return MXQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Per-device cache of the SM count; 0 = not yet queried.
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];

// Checks that the current device is sm_103 and returns its SM count.
int device_check(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MXQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < kMaxDevices) {
    const int cached = g_sms[dev].load(std::memory_order_relaxed);
    if (cached > 0) {
      *num_sms = cached;
      return MXQ_OK;
    }
  }
  int major = 0, minor = 0, sms = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return fail(MXQ_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  if (!mxq_arch_supported(major, minor))
    return fail(MXQ_ERR_ARCH, "device %d is sm_%d%d; libmxq is built for sm_103a only", dev, major,
                minor);
  if (dev >= 0 && dev < kMaxDevices) g_sms[dev].store(sms, std::memory_order_relaxed);
  *num_sms = sms;
  return MXQ_OK;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(MXQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t kgroups(int64_t K) { return (K + mxq::kGroup - 1) / mxq::kGroup; }

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

int mxq::set_error(int status, const char* text) { return fail(status, "%s", text); }

extern "C" {

const char* mxq_status_string(int status) {
  switch (status) {
    case MXQ_OK: return "MXQ_OK";
    case MXQ_ERR_NULL: return "MXQ_ERR_NULL";
    case MXQ_ERR_SHAPE: return "MXQ_ERR_SHAPE";
    case MXQ_ERR_ALIGN: return "MXQ_ERR_ALIGN";
    case MXQ_ERR_UNSUPPORTED: return "MXQ_ERR_UNSUPPORTED";
    case MXQ_ERR_ARCH: return "MXQ_ERR_ARCH";
    case MXQ_ERR_WORKSPACE: return "MXQ_ERR_WORKSPACE";
    case MXQ_ERR_CUDA: return "MXQ_ERR_CUDA";
    default: return "MXQ_ERR_UNKNOWN";
  }
}

const char* mxq_last_error(void) { return g_last_error; }

int mxq_version(void) { return 100; }

int mxq_arch_supported(int major, int minor) { return (major == 10 && minor == 3) ? 1 : 0; }

int mxq_inv_rope_group_quant(const void* x_bf16, int64_t T, int32_t G, int32_t D, int32_t R,
                             const int64_t* pos, const void* cos_bf16, const void* sin_bf16,
                             int64_t cs_ld, int64_t max_pos, uint8_t* q_e4m3, uint8_t* q_e8m0,
                             int32_t* err_flag, mxq_stream_t stream) {
  if (T < 0 || G < 1 || D < 16 || R < 0)
    return fail(MXQ_ERR_SHAPE, "need T >= 0, G >= 1, D >= 16, R >= 0 (T=%lld G=%d D=%d R=%d)",
                (long long)T, G, D, R);
  if (D % 16 != 0) return fail(MXQ_ERR_SHAPE, "D %% 16 != 0 (D=%d)", D);
  // T and T*G first: each factor below 2^31 keeps every product in int64.
  if (T >= (int64_t)1 << 31 || T * G >= (int64_t)1 << 31 || T * G * kgroups(D) >= (int64_t)1 << 31)
    return fail(MXQ_ERR_UNSUPPORTED, "T*G*ceil(D/128) must be < 2^31");
  if (T == 0) return ok();
  if (R > 0) {
    if (R % 16 != 0 || R > 128 || R > D)
      return fail(MXQ_ERR_UNSUPPORTED, "R must be a multiple of 16, <= 128 and <= D (R=%d)", R);
    if (D % 128 != 0)
      return fail(MXQ_ERR_UNSUPPORTED, "R > 0 needs D %% 128 == 0 (D=%d)", D);
    if (max_pos < 1 || cs_ld < R / 2)
      return fail(MXQ_ERR_SHAPE, "need max_pos >= 1 and cs_ld >= R/2 (max_pos=%lld cs_ld=%lld)",
                  (long long)max_pos, (long long)cs_ld);
    if (cs_ld % 8 != 0) return fail(MXQ_ERR_ALIGN, "cs_ld %% 8 != 0 (cs_ld=%lld)", (long long)cs_ld);
    if (!pos || !cos_bf16 || !sin_bf16) return fail(MXQ_ERR_NULL, "pos/cos/sin is NULL with R > 0");
    if (!aligned16(cos_bf16) || !aligned16(sin_bf16) || (reinterpret_cast<uintptr_t>(pos) & 7u))
      return fail(MXQ_ERR_ALIGN, "cos/sin must be 16-byte aligned and pos 8-byte aligned");
  }
  if (!x_bf16 || !q_e4m3 || !q_e8m0) return fail(MXQ_ERR_NULL, "x, q_e4m3 or q_e8m0 is NULL");
  if (!aligned16(x_bf16) || !aligned16(q_e4m3) || !aligned16(q_e8m0))
    return fail(MXQ_ERR_ALIGN, "x, q_e4m3 and q_e8m0 must be 16-byte aligned");
  if (err_flag && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
    return fail(MXQ_ERR_ALIGN, "err_flag must be 4-byte aligned");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::launch_inv_rope_group_quant(x_bf16, T, G, D, R, pos, cos_bf16, sin_bf16,
                                                      cs_ld, max_pos, q_e4m3, q_e8m0, err_flag, sms,
                                                      static_cast<cudaStream_t>(stream)),
                     "inv_rope_group_quant launch");
}

size_t mxq_weight_scale_bytes(int32_t B, int32_t N, int32_t K) {
  if (B < 1 || N < 1 || K < 1) return 0;
  return (size_t)B * kgroups(K) * mxq::sf_row_blocks(N) * mxq::kSfAtomBytes;
}

int mxq_prepare_weight_scales(const uint8_t* w_e8m0, int32_t B, int32_t N, int32_t K,
                              uint8_t* w_sf_prepared, mxq_stream_t stream) {
  if (B < 1 || N < 1 || K < 16 || K % 16 != 0)
    return fail(MXQ_ERR_SHAPE, "need B >= 1, N >= 1, K >= 16, K %% 16 == 0 (B=%d N=%d K=%d)", B, N,
                K);
  if (!w_e8m0 || !w_sf_prepared) return fail(MXQ_ERR_NULL, "w_e8m0 or w_sf_prepared is NULL");
  if (!aligned16(w_e8m0) || !aligned16(w_sf_prepared))
    return fail(MXQ_ERR_ALIGN, "w_e8m0 and w_sf_prepared must be 16-byte aligned");
  if (mxq_weight_scale_bytes(B, N, K) / 4 >= ((size_t)1 << 32))
    return fail(MXQ_ERR_UNSUPPORTED, "prepared scale buffer too large");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::launch_prepare_weight_scales(w_e8m0, B, N, K, w_sf_prepared,
                                                       static_cast<cudaStream_t>(stream)),
                     "prepare_weight_scales launch");
}

size_t mxq_bmm_workspace_bytes(int64_t T, int32_t G, int32_t N, int32_t K) {
  (void)T;
  (void)G;
  (void)N;
  (void)K;
  return 0;
}

static int validate_bmm(const uint8_t* a, const uint8_t* a_sf, const uint8_t* w,
                        const uint8_t* w_sf, void* out, int64_t T, int32_t G, int32_t N,
                        int32_t K) {
  if (T < 0 || G < 1 || N < 16 || K < 16)
    return fail(MXQ_ERR_SHAPE, "need T >= 0, G >= 1, N >= 16, K >= 16 (T=%lld G=%d N=%d K=%d)",
                (long long)T, G, N, K);
  if (K % 16 != 0 || N % 16 != 0)
    return fail(MXQ_ERR_SHAPE, "need K %% 16 == 0 and N %% 16 == 0 (N=%d K=%d)", N, K);
  if (K > 65536) return fail(MXQ_ERR_UNSUPPORTED, "K > 65536");
  if (G > 65535) return fail(MXQ_ERR_UNSUPPORTED, "G > 65535");
  if (T >= ((int64_t)1 << 31) || (int64_t)N * K >= ((int64_t)1 << 40))
    return fail(MXQ_ERR_UNSUPPORTED, "T or N*K too large");
  if (T == 0) return MXQ_OK;
  if (!a || !a_sf || !w || !w_sf || !out) return fail(MXQ_ERR_NULL, "a NULL operand pointer");
  if (!aligned16(a) || !aligned16(a_sf) || !aligned16(w) || !aligned16(w_sf) || !aligned16(out))
    return fail(MXQ_ERR_ALIGN, "operands must be 16-byte aligned");
  return MXQ_OK;
}

int mxq_bmm_a8w8(const uint8_t* a_e4m3, const uint8_t* a_e8m0, const uint8_t* w_e4m3,
                 const uint8_t* w_sf_prepared, void* out_bf16, int64_t T, int32_t G, int32_t N,
                 int32_t K, void* ws, size_t ws_bytes, mxq_stream_t stream) {
  if (int st = validate_bmm(a_e4m3, a_e8m0, w_e4m3, w_sf_prepared, out_bf16, T, G, N, K)) return st;
  const size_t need = mxq_bmm_workspace_bytes(T, G, N, K);
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(MXQ_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, ws_bytes);
  if (T == 0) return ok();
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  const char* why = nullptr;
  cudaError_t e = mxq::launch_bmm_a8w8(a_e4m3, a_e8m0, w_e4m3, w_sf_prepared, out_bf16, T, G, N, K,
                                       sms, static_cast<cudaStream_t>(stream), &why);
  if (e != cudaSuccess && why) return fail(MXQ_ERR_CUDA, "bmm_a8w8: %s", why);
  return cuda_status(e, "bmm_a8w8 launch");
}

size_t mxq_linear_workspace_bytes(int64_t M, int32_t N, int32_t K) {
  if (M < 0 || N < 1 || K < 1) return 0;
  if (M <= mxq::kFusedMaxTokens) return 0;  // one fused launch, no scratch
  if (M >= mxq::kPairMinTokens) return mxq::woa_prefill_layout(M, 1, K).total;
  return round256((size_t)M * K) + round256((size_t)M * kgroups(K)) +
         round256(mxq_bmm_workspace_bytes(M, 1, N, K));
}

int mxq_linear(const void* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_sf_prepared,
               void* out_bf16, int64_t M, int32_t N, int32_t K, void* ws, size_t ws_bytes,
               mxq_stream_t stream) {
  if (M < 0 || N < 16 || K < 16 || K % 16 != 0 || N % 16 != 0)
    return fail(MXQ_ERR_SHAPE, "need M >= 0, N >= 16, K >= 16, N %% 16 == 0, K %% 16 == 0 "
                               "(M=%lld N=%d K=%d)", (long long)M, N, K);
  if (K > 65536) return fail(MXQ_ERR_UNSUPPORTED, "K > 65536");
  if (M >= ((int64_t)1 << 31) || (int64_t)N * K >= ((int64_t)1 << 40))
    return fail(MXQ_ERR_UNSUPPORTED, "M or N*K too large");
  if (M == 0) return ok();
  if (!x_bf16 || !w_e4m3 || !w_sf_prepared || !out_bf16)
    return fail(MXQ_ERR_NULL, "a NULL operand pointer");
  if (!aligned16(x_bf16) || !aligned16(w_e4m3) || !aligned16(w_sf_prepared) || !aligned16(out_bf16))
    return fail(MXQ_ERR_ALIGN, "operands must be 16-byte aligned");
  if (M <= mxq::kFusedMaxTokens) {
    // Few rows: one launch that quantises x inside the GEMM.
    int sms = 0;
    if (int st = device_check(&sms)) return st;
    const char* why = nullptr;
    cudaError_t e = mxq::launch_wo_a_fused(x_bf16, nullptr, nullptr, nullptr, 0, 0, 0, w_e4m3,
                                           w_sf_prepared, out_bf16, M, 1, N, K, nullptr, sms,
                                           static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess && why) return fail(MXQ_ERR_CUDA, "linear: %s", why);
    return cuda_status(e, "linear (fused) launch");
  }
  const size_t need = mxq_linear_workspace_bytes(M, N, K);
  if (!ws || ws_bytes < need)
    return fail(MXQ_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, ws_bytes);
  if (!aligned16(ws)) return fail(MXQ_ERR_ALIGN, "workspace must be 16-byte aligned");
  if (M >= mxq::kPairMinTokens) {
    // Many rows: one launch of the CTA-pair GEMM whose warps quantise x.
    if (M * kgroups(K) >= (int64_t)1 << 31)
      return fail(MXQ_ERR_UNSUPPORTED, "M*ceil(K/128) must be < 2^31");
    int sms = 0;
    if (int st = device_check(&sms)) return st;
    const char* why = nullptr;
    cudaError_t e = mxq::launch_wo_a_prefill(x_bf16, nullptr, nullptr, nullptr, 0, 0, 0, w_e4m3,
                                             w_sf_prepared, out_bf16, M, 1, N, K, nullptr, ws, sms,
                                             static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess && why) return fail(MXQ_ERR_CUDA, "linear: %s", why);
    return cuda_status(e, "linear (quantising pair form) launch");
  }
  uint8_t* codes = static_cast<uint8_t*>(ws);
  uint8_t* scales = codes + round256((size_t)M * K);
  uint8_t* gemm_ws = scales + round256((size_t)M * kgroups(K));
  if (int st = mxq_inv_rope_group_quant(x_bf16, M, 1, K, 0, nullptr, nullptr, nullptr, 0, 0, codes,
                                        scales, nullptr, stream))
    return st;
  return mxq_bmm_a8w8(codes, scales, w_e4m3, w_sf_prepared, out_bf16, M, 1, N, K, gemm_ws,
                      ws_bytes - (size_t)(gemm_ws - codes), stream);
}

size_t mxq_wo_a_workspace_bytes(int64_t T, int32_t G, int32_t D, int32_t N) {
  (void)N;
  if (T < 0 || G < 1 || D < 1) return 0;
  if (T <= mxq::kFusedMaxTokens) return 0;
  if (T >= mxq::kPairMinTokens) return mxq::woa_prefill_layout(T, G, D).total;
  return round256((size_t)T * G * D) + round256((size_t)T * G * kgroups(D));
}

int mxq_wo_a(const void* x_bf16, const int64_t* pos, const void* cos_bf16, const void* sin_bf16,
             int64_t cs_ld, int64_t max_pos, const uint8_t* w_e4m3, const uint8_t* w_sf_prepared,
             void* out_bf16, int64_t T, int32_t G, int32_t D, int32_t N, int32_t R,
             int32_t* err_flag, void* ws, size_t ws_bytes, mxq_stream_t stream) {
  // Same argument rules as mxq_inv_rope_group_quant followed by mxq_bmm_a8w8.
  if (T < 0 || G < 1 || D < 16 || R < 0 || N < 16)
    return fail(MXQ_ERR_SHAPE, "need T >= 0, G >= 1, D >= 16, R >= 0, N >= 16");
  if (D % 16 != 0 || N % 16 != 0) return fail(MXQ_ERR_SHAPE, "need D %% 16 == 0 and N %% 16 == 0");
  if (D > 65536 || G > 65535) return fail(MXQ_ERR_UNSUPPORTED, "D > 65536 or G > 65535");
  if (T >= ((int64_t)1 << 31) || (int64_t)N * D >= ((int64_t)1 << 40))
    return fail(MXQ_ERR_UNSUPPORTED, "T or N*D too large");
  if (T == 0) return ok();
  if (R > 0) {
    if (R % 16 != 0 || R > 128 || R > D)
      return fail(MXQ_ERR_UNSUPPORTED, "R must be a multiple of 16, <= 128 and <= D (R=%d)", R);
    if (D % 128 != 0) return fail(MXQ_ERR_UNSUPPORTED, "R > 0 needs D %% 128 == 0 (D=%d)", D);
    if (max_pos < 1 || cs_ld < R / 2)
      return fail(MXQ_ERR_SHAPE, "need max_pos >= 1 and cs_ld >= R/2");
    if (cs_ld % 8 != 0) return fail(MXQ_ERR_ALIGN, "cs_ld %% 8 != 0");
    if (!pos || !cos_bf16 || !sin_bf16) return fail(MXQ_ERR_NULL, "pos/cos/sin is NULL with R > 0");
    if (!aligned16(cos_bf16) || !aligned16(sin_bf16) || (reinterpret_cast<uintptr_t>(pos) & 7u))
      return fail(MXQ_ERR_ALIGN, "cos/sin must be 16-byte aligned and pos 8-byte aligned");
  }
  if (!x_bf16 || !w_e4m3 || !w_sf_prepared || !out_bf16)
    return fail(MXQ_ERR_NULL, "a NULL operand pointer");
  if (!aligned16(x_bf16) || !aligned16(w_e4m3) || !aligned16(w_sf_prepared) || !aligned16(out_bf16))
    return fail(MXQ_ERR_ALIGN, "operands must be 16-byte aligned");
  if (err_flag && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
    return fail(MXQ_ERR_ALIGN, "err_flag must be 4-byte aligned");
  if (T <= mxq::kFusedMaxTokens) {
    int sms = 0;
    if (int st = device_check(&sms)) return st;
    const char* why = nullptr;
    cudaError_t e = mxq::launch_wo_a_fused(x_bf16, pos, cos_bf16, sin_bf16, cs_ld, max_pos, R,
                                           w_e4m3, w_sf_prepared, out_bf16, T, G, N, D, err_flag,
                                           sms, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess && why) return fail(MXQ_ERR_CUDA, "wo_a: %s", why);
    return cuda_status(e, "wo_a (fused) launch");
  }
  const size_t need = mxq_wo_a_workspace_bytes(T, G, D, N);
  if (!ws || ws_bytes < need)
    return fail(MXQ_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, ws_bytes);
  if (!aligned16(ws)) return fail(MXQ_ERR_ALIGN, "workspace must be 16-byte aligned");
  if (T >= mxq::kPairMinTokens) {
    if (T * G * kgroups(D) >= (int64_t)1 << 31)
      return fail(MXQ_ERR_UNSUPPORTED, "T*G*ceil(D/128) must be < 2^31");
    int sms = 0;
    if (int st = device_check(&sms)) return st;
    const char* why = nullptr;
    cudaError_t e = mxq::launch_wo_a_prefill(x_bf16, pos, cos_bf16, sin_bf16, cs_ld, max_pos, R,
                                             w_e4m3, w_sf_prepared, out_bf16, T, G, N, D, err_flag,
                                             ws, sms, static_cast<cudaStream_t>(stream), &why);
    if (e != cudaSuccess && why) return fail(MXQ_ERR_CUDA, "wo_a: %s", why);
    return cuda_status(e, "wo_a (quantising pair form) launch");
  }
  uint8_t* codes = static_cast<uint8_t*>(ws);
  uint8_t* scales = codes + round256((size_t)T * G * D);
  if (int st = mxq_inv_rope_group_quant(x_bf16, T, G, D, R, pos, cos_bf16, sin_bf16, cs_ld, max_pos,
                                        codes, scales, err_flag, stream))
    return st;
  return mxq_bmm_a8w8(codes, scales, w_e4m3, w_sf_prepared, out_bf16, T, G, N, D, nullptr, 0,
                      stream);
}

int mxq_dequant_bf16(const uint8_t* w_e4m3, const uint8_t* w_e8m0, void* out_bf16, int32_t B,
                     int32_t N, int32_t K, mxq_stream_t stream) {
  if (B < 0 || N < 0 || K < 16 || K % 16 != 0)
    return fail(MXQ_ERR_SHAPE, "need B >= 0, N >= 0, K >= 16, K %% 16 == 0 (B=%d N=%d K=%d)", B, N,
                K);
  if ((int64_t)B * N * (K / 16) >= ((int64_t)1 << 32))
    return fail(MXQ_ERR_UNSUPPORTED, "B*N*K/16 must be < 2^32");
  if (B == 0 || N == 0) return ok();
  if (!w_e4m3 || !w_e8m0 || !out_bf16) return fail(MXQ_ERR_NULL, "a NULL operand pointer");
  if (!aligned16(w_e4m3) || !aligned16(w_e8m0) || !aligned16(out_bf16))
    return fail(MXQ_ERR_ALIGN, "operands must be 16-byte aligned");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::launch_dequant_bf16(w_e4m3, w_e8m0, out_bf16, B, N, K, sms,
                                              static_cast<cudaStream_t>(stream)),
                     "dequant_bf16 launch");
}

int mxq_scales_f32_to_e8m0(const float* s, int64_t n, uint8_t* out, int32_t* err_flag,
                           mxq_stream_t stream) {
  if (n < 0) return fail(MXQ_ERR_SHAPE, "n < 0");
  if (n == 0) return ok();
  if (!s || !out) return fail(MXQ_ERR_NULL, "s or out is NULL");
  if (!aligned16(s) || !aligned16(out)) return fail(MXQ_ERR_ALIGN, "s and out must be 16-byte aligned");
  if (err_flag && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
    return fail(MXQ_ERR_ALIGN, "err_flag must be 4-byte aligned");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::launch_scales_f32_to_e8m0(s, n, out, err_flag,
                                                    static_cast<cudaStream_t>(stream)),
                     "scales_f32_to_e8m0 launch");
}

int mxq_rope_kv_insert(const void* q_bf16, void* q_out_bf16, int64_t T, int32_t H, int32_t Dq,
                       const void* kv_bf16, int32_t Dk, const int64_t* pos, const void* cos_bf16,
                       const void* sin_bf16, int64_t cs_ld, int64_t max_pos, int32_t R,
                       const int64_t* slot_mapping, void* kv_cache, int64_t num_slots,
                       int32_t cache_dtype, const float* kv_scale, int32_t* err_flag,
                       mxq_stream_t stream) {
  if (T < 0 || H < 0 || Dk < 16 || R < 0 || num_slots < 0 || (H > 0 && Dq < 16))
    return fail(MXQ_ERR_SHAPE, "need T >= 0, H >= 0, Dk >= 16, R >= 0, num_slots >= 0, "
                               "Dq >= 16 when H > 0 (T=%lld H=%d Dq=%d Dk=%d R=%d)",
                (long long)T, H, Dq, Dk, R);
  if (Dk % 16 != 0 || (H > 0 && Dq % 16 != 0))
    return fail(MXQ_ERR_SHAPE, "need Dk %% 16 == 0 and Dq %% 16 == 0 (Dq=%d Dk=%d)", Dq, Dk);
  if (cache_dtype != MXQ_CACHE_E4M3 && cache_dtype != MXQ_CACHE_BF16)
    return fail(MXQ_ERR_UNSUPPORTED, "cache_dtype must be MXQ_CACHE_E4M3 or MXQ_CACHE_BF16");
  if (R % 16 != 0 || R > Dk || (H > 0 && R > Dq))
    return fail(MXQ_ERR_UNSUPPORTED, "R must be a multiple of 16, <= Dk and <= Dq (R=%d)", R);
  // Every factor is below 2^31 here, so the products fit in int64.
  if (T >= ((int64_t)1 << 31) ||
      T * ((int64_t)H * (Dq / 8) + Dk / 8) >= ((int64_t)1 << 31))
    return fail(MXQ_ERR_UNSUPPORTED, "T*H*Dq/8 + T*Dk/8 must be < 2^31");
  if (T == 0) return ok();
  if (R > 0) {
    if (max_pos < 1 || cs_ld < R / 2)
      return fail(MXQ_ERR_SHAPE, "need max_pos >= 1 and cs_ld >= R/2 (max_pos=%lld cs_ld=%lld)",
                  (long long)max_pos, (long long)cs_ld);
    if (cs_ld % 8 != 0) return fail(MXQ_ERR_ALIGN, "cs_ld %% 8 != 0 (cs_ld=%lld)", (long long)cs_ld);
    if (!pos || !cos_bf16 || !sin_bf16) return fail(MXQ_ERR_NULL, "pos/cos/sin is NULL with R > 0");
    if (!aligned16(cos_bf16) || !aligned16(sin_bf16) || (reinterpret_cast<uintptr_t>(pos) & 7u))
      return fail(MXQ_ERR_ALIGN, "cos/sin must be 16-byte aligned and pos 8-byte aligned");
  }
  if (!kv_bf16 || !slot_mapping || !kv_cache) return fail(MXQ_ERR_NULL, "kv, slot_mapping or kv_cache is NULL");
  if (H > 0 && (!q_bf16 || !q_out_bf16)) return fail(MXQ_ERR_NULL, "q or q_out is NULL with H > 0");
  if (cache_dtype == MXQ_CACHE_E4M3 && !kv_scale) return fail(MXQ_ERR_NULL, "kv_scale is NULL for an E4M3 cache");
  if (!aligned16(kv_bf16) || !aligned16(kv_cache) || (H > 0 && (!aligned16(q_bf16) || !aligned16(q_out_bf16))))
    return fail(MXQ_ERR_ALIGN, "q, q_out, kv and kv_cache must be 16-byte aligned");
  if (H > 0 && q_bf16 != q_out_bf16) {
    // Distinct query buffers must not overlap (in place is q_out == q exactly).
    const uintptr_t a = reinterpret_cast<uintptr_t>(q_bf16), b = reinterpret_cast<uintptr_t>(q_out_bf16);
    const uintptr_t n = (uintptr_t)T * (uintptr_t)H * (uintptr_t)Dq * 2u;
    if (a < b + n && b < a + n)
      return fail(MXQ_ERR_SHAPE, "q_out overlaps q without being q itself");
  }
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) ||
      (kv_scale && (reinterpret_cast<uintptr_t>(kv_scale) & 3u)) ||
      (err_flag && (reinterpret_cast<uintptr_t>(err_flag) & 3u)))
    return fail(MXQ_ERR_ALIGN, "slot_mapping must be 8-byte aligned, kv_scale and err_flag 4-byte aligned");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(
      mxq::launch_rope_kv_insert(q_bf16, q_out_bf16, T, H, Dq, kv_bf16, Dk, pos, cos_bf16, sin_bf16,
                                 cs_ld, max_pos, R, slot_mapping, kv_cache, num_slots,
                                 cache_dtype == MXQ_CACHE_E4M3 ? 1 : 0, kv_scale, err_flag, sms,
                                 static_cast<cudaStream_t>(stream)),
      "rope_kv_insert launch");
}

int mxq_debug_set_pair_limit(int pairs) { return mxq::set_pair_limit(pairs); }

int mxq_debug_set_lazy_pairs(int from) {
  const int prev = mxq::set_lazy_pairs(from);
  return prev >= (1 << 30) ? -1 : prev;
}

int mxq_debug_takeovers(uint32_t* host_value, int clear) {
  if (!host_value) return fail(MXQ_ERR_NULL, "host_value is NULL");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::takeover_count(host_value, clear != 0), "takeover count read");
}

int mxq_watchdog_read(uint32_t* host_value, int clear) {
  if (!host_value) return fail(MXQ_ERR_NULL, "host_value is NULL");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::watchdog_read(host_value, clear != 0), "watchdog read");
}

int mxq_watchdog_selftest(uint64_t limit_ns, mxq_stream_t stream) {
  if (limit_ns < 1 || limit_ns > 2000000000ull)
    return fail(MXQ_ERR_SHAPE, "limit_ns must be in [1, 2e9]");
  int sms = 0;
  if (int st = device_check(&sms)) return st;
  return cuda_status(mxq::launch_watchdog_selftest(limit_ns, static_cast<cudaStream_t>(stream)),
                     "watchdog self-test launch");
}

}  // extern "C"
