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
//
// A large query rotated out of place is a copy of which one part in Dq/R
// changes: it runs in a streaming kernel of bulk copies instead (blocks of
// whole query rows through shared memory, rotated there), which keeps far
// more bytes in flight per SM than one 16-byte chunk per thread; the KV rows
// then run through the item kernel alone (measured: doing their items
// inside the streaming kernel, first or one per thread and block, made the
// 8K-token call 184 us instead of 169 us).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "mxq.h"
#include "mxq_internal.h"
#include "mxq_ptx.cuh"
#include "quant_common.cuh"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

// Streaming query kernel: 3 stages of up to 32 KB of whole rows per CTA, two
// CTAs per SM (192 KB of copies in flight per SM).
constexpr int kBulkThreads = 128;
constexpr int kBulkStages = 3;
constexpr int kBulkStageBytes = 32 * 1024;
constexpr int kBulkCtasPerSm = 2;
constexpr uint64_t kBulkWaitNs = 4000000000ull;
constexpr uint32_t kWdKvBulk = 32;  // watchdog bit of this kernel
// Out-of-place queries of at least this many bytes (about four blocks per
// CTA) take the streaming kernel; below that a second launch and blocks that
// find no pipeline to fill cost more than they save (measured: q [64, 64,
// 512] 4.2 us per call in the item kernel, 5.9 us streamed).
constexpr int64_t kBulkMinBytes = 32 << 20;

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

// Forward rotation of one rotate-half pair of chunks (x0 in the lower half,
// x1 in the upper) with the cos/sin entries j..j+7 of position p: one
// rounding per value, as the oracle.
__device__ __forceinline__ void rope_pair(const uint4& va, const uint4& vb, const uint4& cw,
                                          const uint4& sw, float (&y0)[8], float (&y1)[8]) {
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

// One work item of the row kernels (see the top of the file).
__device__ __forceinline__ void kv_item(const KvArgs& a, uint32_t it, float scale) {
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
    if (sl < 0 || over || bad) return;
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
    return;
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
    rope_pair(va, vb, cw, sw, y0, y1);
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

__global__ void __launch_bounds__(kThreads, kBlocksPerSm) rope_kv_insert_kernel(const KvArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Everything below reads what preceding kernels wrote.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float scale = a.fp8 ? __ldg(a.scale) : 1.0f;
  const uint32_t stride = gridDim.x * kThreads;
  for (uint32_t it = blockIdx.x * kThreads + threadIdx.x; it < a.n_items; it += stride)
    kv_item(a, it, scale);
}

struct QBulkArgs {
  const uint8_t* q;
  uint8_t* q_out;
  const int64_t* pos;
  const uint16_t* cos_tab;
  const uint16_t* sin_tab;
  int64_t cs_ld, max_pos;
  int64_t rows;   // T * H query rows of Dq values
  int64_t units;  // blocks of U consecutive rows (the last may be shorter)
  int H, Dq, R, U;
  uint32_t* watchdog;
};

// Query rows out of place: each CTA walks units u = blockIdx.x, + gridDim.x,
// ...; a unit's rows are copied into a shared-memory stage with one bulk copy,
// their rotated slices are rewritten there (zeros for a token with an
// invalid position), and the stage goes back to q_out with one bulk copy.
// Three stages per CTA: the copy of a stage is issued again as soon as the
// store of the unit before the current one has read it.
__global__ void __launch_bounds__(kBulkThreads) rope_q_bulk_kernel(const QBulkArgs a) {
  extern __shared__ __align__(128) uint8_t stages[];
  __shared__ uint64_t full[kBulkStages];
  const int tid = threadIdx.x;
  const size_t row_bytes = (size_t)a.Dq * 2;
  if (tid == 0) {
    for (int s = 0; s < kBulkStages; ++s) ptx::mbar_init(&full[s], 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The query and the positions come from preceding kernels.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t u0 = blockIdx.x;
  const int64_t ustep = gridDim.x;
  auto unit_rows = [&](int64_t u) { return (int)min((int64_t)a.U, a.rows - u * a.U); };
  auto issue = [&](int64_t u, int s) {
    const uint32_t bytes = (uint32_t)(unit_rows(u) * row_bytes);
    ptx::mbar_arrive_expect_tx(&full[s], bytes);
    ptx::bulk_load(stages + s * kBulkStageBytes, a.q + (size_t)u * a.U * row_bytes, bytes, &full[s]);
  };
  if (tid == 0)
    for (int s = 0; s < kBulkStages; ++s)
      if (u0 + s * ustep < a.units) issue(u0 + s * ustep, s);
  const int half = a.R / 16;            // rotate-half chunk pairs per row
  const int c_first = (a.Dq - a.R) / 8;  // first chunk of the rotated slice
  int k = 0;
  for (int64_t u = u0; u < a.units; u += ustep, ++k) {
    const int s = k % kBulkStages;
    const bool ok = ptx::mbar_wait(&full[s], (uint32_t)(k / kBulkStages) & 1u, kBulkWaitNs);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicOr(a.watchdog, kWdKvBulk);
      break;
    }
    uint8_t* st = stages + s * kBulkStageBytes;
    const int nr = unit_rows(u);
    for (int item = tid; item < nr * half; item += kBulkThreads) {
      const int rl = item / half;
      const int pr = item - rl * half;
      const int64_t t = (u * a.U + rl) / a.H;
      const int64_t p = __ldg(a.pos + t);
      uint4* rp = reinterpret_cast<uint4*>(st + (size_t)rl * row_bytes);
      const int c0 = c_first + pr;
      const int c1 = c0 + half;
      float y0[8], y1[8];
      if (p < 0 || p >= a.max_pos) {
#pragma unroll
        for (int e = 0; e < 8; ++e) y0[e] = y1[e] = 0.0f;
      } else {
        const uint4 cw = __ldg(reinterpret_cast<const uint4*>(a.cos_tab + p * a.cs_ld + pr * 8));
        const uint4 sw = __ldg(reinterpret_cast<const uint4*>(a.sin_tab + p * a.cs_ld + pr * 8));
        rope_pair(rp[c0], rp[c1], cw, sw, y0, y1);
      }
      rp[c0] = to_bf16x8(y0);
      rp[c1] = to_bf16x8(y1);
    }
    ptx::fence_proxy_async_smem();  // the rotated chunks before the copy reads them
    __syncthreads();
    if (tid == 0) {
      ptx::bulk_store(a.q_out + (size_t)u * a.U * row_bytes, st, (uint32_t)(nr * row_bytes));
      ptx::bulk_commit_group();
      // The store of the previous unit has read its stage: refill that stage.
      if (k >= 1) {
        const int64_t un = u + (kBulkStages - 1) * ustep;
        if (un < a.units) {
          ptx::bulk_wait_read<1>();
          issue(un, (k - 1) % kBulkStages);
        }
      }
    }
  }
  if (tid == 0) ptx::bulk_wait_all();  // the stores are done before the stages go away
}

cudaError_t launch_rope_q_bulk(QBulkArgs b, int num_sms, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Per device, once: the shared-memory opt-in and the watchdog's address.
  static std::atomic<uint64_t> ready{0};
  static uint32_t* wd[64];
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(rope_q_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBulkStages * kBulkStageBytes);
    if (e != cudaSuccess) return e;
    e = watchdog_address(&wd[dev & 63]);
    if (e != cudaSuccess) return e;
    ready.fetch_or(bit, std::memory_order_acq_rel);
  }
  b.watchdog = wd[dev & 63];
  const int64_t cap = (int64_t)num_sms * kBulkCtasPerSm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(b.units < cap ? b.units : cap), 1, 1);
  cfg.blockDim = dim3(kBulkThreads, 1, 1);
  cfg.dynamicSmemBytes = kBulkStages * kBulkStageBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rope_q_bulk_kernel, b);
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
  const bool streamed = H > 0 && q != q_out && T * H * (int64_t)Dq * 2 >= kBulkMinBytes &&
                        Dq * 2 <= kBulkStageBytes;
  // The item kernel's query part (none when the query is streamed; in place,
  // the query's chunks outside the slice stay where they are).
  const int hq = streamed ? 0 : H;
  a.pq = (hq > 0 && q != q_out) ? (uint32_t)((Dq - R) / 8) : 0u;
  a.pk = (uint32_t)((Dk - R) / 8);
  a.iq = a.pq + (uint32_t)(R / 16);
  a.ik = a.pk + (uint32_t)(R / 16);
  a.q_items = (uint32_t)(T * hq) * a.iq;
  a.n_items = a.q_items + (uint32_t)T * a.ik;
  if (streamed) {
    // A large query out of place: the streaming kernel, then the KV rows.
    QBulkArgs b = {};
    b.q = static_cast<const uint8_t*>(q);
    b.q_out = static_cast<uint8_t*>(q_out);
    b.pos = pos;
    b.cos_tab = a.cos_tab;
    b.sin_tab = a.sin_tab;
    b.cs_ld = cs_ld;
    b.max_pos = max_pos;
    b.rows = T * H;
    b.H = H;
    b.Dq = Dq;
    b.R = R;
    b.U = kBulkStageBytes / (Dq * 2);  // at least one row
    b.units = ceil_div(b.rows, b.U);
    cudaError_t e = launch_rope_q_bulk(b, num_sms, s);
    if (e != cudaSuccess) return e;
  }
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
