// mxq_linear_noalloc: the MXFP8 linear layer for callers that cannot
// allocate device memory.
//
// mxq_linear needs a caller-provided workspace for the quantised activation
// (E4M3 codes and E8M0 scale bytes of x).  Some callers have no way to
// provide one: a plain-C or embedded host program that links only this
// library and holds no device allocator, or a latency-critical serving loop
// that must never call cudaMalloc/cudaFree (both can synchronise the device)
// and whose device memory was reserved once at start-up by somebody else.
// This entry point takes the workspace from a fixed array in the library's
// own device memory instead, so it allocates nothing.
//
// The array is a file-scope __device__ variable of MXQ_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads the library keeps it until the process exits.
// Host code may not use the variable's name as a device address (on the host
// it names a shadow object), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// the device.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MXQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<uint8_t*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Device address of the scratch array on the current device (looked up once
// per device); nullptr and a status on failure.
int scratch_on_current_device(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mxq::set_error(MXQ_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return mxq::set_error(MXQ_ERR_UNSUPPORTED, "device index >= 64");
  uint8_t* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess || addr == nullptr)
        return mxq::set_error(MXQ_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                             : "scratch symbol has no address");
      p = static_cast<uint8_t*>(addr);
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return MXQ_OK;
}

}  // namespace

extern "C" int mxq_linear_noalloc(const void* x_bf16, const uint8_t* w_e4m3,
                                  const uint8_t* w_sf_prepared, void* out_bf16, int64_t M,
                                  int32_t N, int32_t K, mxq_stream_t stream) {
  // Every argument rule of mxq_linear, checked before anything is enqueued.
  if (M < 0 || N < 16 || K < 16 || K % 16 != 0 || N % 16 != 0)
    return mxq::set_error(MXQ_ERR_SHAPE, "need M >= 0, N >= 16, K >= 16, N % 16 == 0, K % 16 == 0");
  if (K > 65536) return mxq::set_error(MXQ_ERR_UNSUPPORTED, "K > 65536");
  if (M >= ((int64_t)1 << 31) || (int64_t)N * K >= ((int64_t)1 << 40))
    return mxq::set_error(MXQ_ERR_UNSUPPORTED, "M or N*K too large");
  if (M == 0) return mxq::set_error(MXQ_OK, "");
  if (!x_bf16 || !w_e4m3 || !w_sf_prepared || !out_bf16)
    return mxq::set_error(MXQ_ERR_NULL, "a NULL operand pointer");
  if (((reinterpret_cast<uintptr_t>(x_bf16) | reinterpret_cast<uintptr_t>(w_e4m3) |
        reinterpret_cast<uintptr_t>(w_sf_prepared) | reinterpret_cast<uintptr_t>(out_bf16)) &
       15u) != 0)
    return mxq::set_error(MXQ_ERR_ALIGN, "operands must be 16-byte aligned");
  // Up to 32 rows the linear is one launch that quantises x inside the GEMM
  // and needs no scratch at all.
  if (M <= mxq::kFusedMaxTokens)
    return mxq_linear(x_bf16, w_e4m3, w_sf_prepared, out_bf16, M, N, K, nullptr, 0, stream);
  // Scratch layout: codes [M, K] (256-byte aligned), then scale bytes [M, ceil(K/128)].
  const size_t codes_bytes = round256((size_t)M * (size_t)K);
  const size_t scale_bytes = round256((size_t)M * (size_t)((K + 127) / 128));
  if ((size_t)M > MXQ_NOALLOC_SCRATCH_BYTES || codes_bytes + scale_bytes > MXQ_NOALLOC_SCRATCH_BYTES)
    return mxq::set_error(MXQ_ERR_WORKSPACE,
                          "M*K too large for the fixed scratch of mxq_linear_noalloc "
                          "(MXQ_NOALLOC_SCRATCH_BYTES); use mxq_linear with a workspace");
  uint8_t* scratch = nullptr;
  if (int st = scratch_on_current_device(&scratch)) return st;
  uint8_t* codes = scratch;
  uint8_t* scales = scratch + codes_bytes;
  // Both stages overwrite every scratch byte they later read, so nothing has
  // to be cleared between calls.  The arguments of both calls were checked
  // above, so neither returns an argument error after the first has been
  // enqueued.
  if (int st = mxq_inv_rope_group_quant(x_bf16, M, 1, K, 0, nullptr, nullptr, nullptr, 0, 0, codes,
                                        scales, nullptr, stream))
    return st;
  return mxq_bmm_a8w8(codes, scales, w_e4m3, w_sf_prepared, out_bf16, M, 1, N, K, nullptr, 0,
                      stream);
}
