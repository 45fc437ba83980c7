// Block-scaled batched a8w8 GEMM on the 5th-generation tensor cores.
//
// Page "[ROCm][DSV4][Perf] Use FP8 WO_A output projection", Summary item 2:
// an MX-scale batched GEMM that consumes the quantised activation and the
// checkpoint's native FP8 weight.  Page "[ROCm][DSv4.1][Perf] Dequantize the
// MXFP8 weight once when dot_scaled cannot be used", Purpose: K % 128 != 0
// (K = 576, 288) must work without dequantising the weight per call.
//
//   out[t, g, n] = bf16( sum_k A[t,g,k] * W[g,n,k] ),
//   A = E4M3(a) * 2^(sa-127), W = E4M3(w) * 2^(sw-127), one scale per 128 k.
//
// Design (one CTA = one 128 x BN output tile of one group g, optionally one
// K-slice of it):
//   warp 0      producer: TMA (128B-swizzled) loads of the A and W tiles for
//               one 128-wide K group per pipeline stage, a bulk copy of the
//               prepared weight-scale atom(s), and a gather of the
//               activation scale bytes into the same 512-byte atom layout.
//   warp 1      TMEM owner and MMA issuer: per stage, tcgen05.cp of the scale
//               atoms into TMEM, then four tcgen05.mma kind::mxf8f6f4
//               block_scale (K = 32 each; the group's byte is replicated in
//               all four bytes of its word, so every 32-block sees the
//               group scale), then tcgen05.commit to free the stage.
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator, RNE to BF16,
//               stores.
// The K tail is the TMA's zero fill past K.  Two orientations:
//   normal  (many tokens): MMA M = 128 tokens, MMA N = BN weight rows.
//   swapped (few tokens):  MMA M = 128 weight rows, MMA N = BN tokens, so the
//               weight streams through the tensor cores with no padding of
//               the token axis to 128.  The K range may be split over the
//               CTAs of a thread-block cluster, whose fp32 partial tiles are
//               summed in rank order through distributed shared memory
//               (deterministic, no global workspace).
// Every wait is bounded in wall time; on expiry the kernel sets a watchdog
// bit, drains its own copies, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"
#include "mxq_ptx.cuh"

namespace mxq {

__device__ uint32_t g_watchdog;

namespace {

constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr uint32_t kWdProducer = 1, kWdMma = 2, kWdEpilogue = 4, kWdDrain = 8;
constexpr int kThreads = 192;

struct BmmArgs {
  const uint8_t* a_sf;  // [T][G][KG]
  const uint8_t* w_sf;  // prepared: [G][KG][NB][512]
  __nv_bfloat16* out;   // [T][G][N]
  int T, G, N, K, KG, NB;
  int x_tiles, y_tiles;
  int splits, kg_per_split;
};

template <bool SWAP, int BN, int NSTAGE>
struct Cfg {
  static constexpr int BM = 128;
  static constexpr int BK = 128;
  static constexpr int Y_ATOMS = (BN + 127) / 128;
  static constexpr int ACT_ATOMS = SWAP ? Y_ATOMS : 1;
  static constexpr int X_TILE = BM * BK;
  static constexpr int Y_TILE = BN * BK;
  static constexpr int SFX_BYTES = kSfAtomBytes;
  static constexpr int SFY_BYTES = Y_ATOMS * kSfAtomBytes;
  static constexpr int W_SF_BYTES = (SWAP ? 1 : Y_ATOMS) * kSfAtomBytes;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_Y = OFF_X + NSTAGE * X_TILE;
  static constexpr int OFF_SFX = OFF_Y + NSTAGE * Y_TILE;
  static constexpr int OFF_SFY = OFF_SFX + NSTAGE * SFX_BYTES;
  static constexpr int OFF_BAR = OFF_SFY + NSTAGE * SFY_BYTES;
  static constexpr int N_BARS = 2 * NSTAGE + 1;
  static constexpr int OFF_SLOT = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_SLOT + 16 + 1024;
  static constexpr int SF_COLS = 4 + 4 * Y_ATOMS;
  static constexpr int TMEM_USED = BN + NSTAGE * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                   : TMEM_USED <= 64  ? 64
                                   : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256
                                                      : 512;
  static constexpr int PART_PITCH = BN + 1;  // fp32 partial tile [128][BN+1] (aliases stages)
  // Instruction descriptor, kind::mxf8f6f4 with block scaling: E4M3 A and
  // B (format 0), both K-major, N >> 3 at bits 17-22, UE8M0 scale type at
  // bit 23, M >> 4 at bits 24-28, scale-factor ids 0.
  static constexpr uint32_t IDESC =
      (1u << 23) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(128 * PART_PITCH * 4 <= OFF_BAR, "partial tile must fit in the stage buffers");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
};

__device__ __forceinline__ void watchdog(volatile int* abort_flag, uint32_t bit) {
  *abort_flag = 1;
  atomicOr(&g_watchdog, bit);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&r);
}

template <bool SWAP, int BN, int NSTAGE>
__global__ void __launch_bounds__(kThreads, 1)
    bmm_a8w8_kernel(const __grid_constant__ CUtensorMap tm_act,
                    const __grid_constant__ CUtensorMap tm_w, const BmmArgs p) {
  using C = Cfg<SWAP, BN, NSTAGE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NSTAGE;
  uint64_t* acc_full = empty + NSTAGE;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SLOT);
  __shared__ int abort_shared;
  volatile int* abort_flag = &abort_shared;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.splits;
  const int tile = blockIdx.x / p.splits;
  const int g = blockIdx.y;
  const int x0 = (tile % p.x_tiles) * C::BM;  // first row of the MMA-A operand
  const int y0 = (tile / p.x_tiles) * BN;     // first row of the MMA-B operand
  const int kg_begin = split * p.kg_per_split;
  const int kg_end = min(p.KG, kg_begin + p.kg_per_split);
  const int nk = max(0, kg_end - kg_begin);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      ptx::mbar_init(&full[s], 2);  // producer's expect_tx arrival + scale-gather arrival
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(acc_full, 1);
    abort_shared = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_act);
    ptx::prefetch_tmap(&tm_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Activation scale rows handled by this lane: atom a, word j <-> row
    // a*128 + 32*j + lane of the activation operand.
    const int act_rows = SWAP ? BN : C::BM;
    const int act_row0 = SWAP ? y0 : x0;
    uint32_t words[4 * C::ACT_ATOMS];
    auto gather = [&](int kg) {
#pragma unroll
      for (int a = 0; a < C::ACT_ATOMS; ++a)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = a * 128 + 32 * j + lane;
          const int t = act_row0 + r;
          uint32_t b = 127u;
          if (r < act_rows && t < p.T) b = __ldg(p.a_sf + ((size_t)t * p.G + g) * p.KG + kg);
          words[a * 4 + j] = b * 0x01010101u;
        }
    };
    int issued = 0;
    if (nk > 0) gather(kg_begin);
    for (int it = 0; it < nk; ++it) {
      const int s = it % NSTAGE;
      const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
      if (*abort_flag) break;
      if (!ptx::mbar_wait(&empty[s], ph ^ 1u, kWaitLimitNs)) {
        watchdog(abort_flag, kWdProducer);
        break;
      }
      const int kg = kg_begin + it;
      uint8_t* xs = smem + C::OFF_X + s * C::X_TILE;
      uint8_t* ys = smem + C::OFF_Y + s * C::Y_TILE;
      uint8_t* sfx = smem + C::OFF_SFX + s * C::SFX_BYTES;
      uint8_t* sfy = smem + C::OFF_SFY + s * C::SFY_BYTES;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(&full[s], C::X_TILE + C::Y_TILE + C::W_SF_BYTES);
        if (!SWAP) {
          ptx::tma_load_3d(xs, &tm_act, &full[s], kg * 128, g, x0);
          ptx::tma_load_3d(ys, &tm_w, &full[s], kg * 128, y0, g);
          ptx::bulk_load(sfy, p.w_sf + (((size_t)g * p.KG + kg) * p.NB + y0 / 128) * kSfAtomBytes,
                         C::W_SF_BYTES, &full[s]);
        } else {
          ptx::tma_load_3d(xs, &tm_w, &full[s], kg * 128, x0, g);
          ptx::tma_load_3d(ys, &tm_act, &full[s], kg * 128, g, y0);
          ptx::bulk_load(sfx, p.w_sf + (((size_t)g * p.KG + kg) * p.NB + x0 / 128) * kSfAtomBytes,
                         C::W_SF_BYTES, &full[s]);
        }
      }
      uint8_t* act_sf = SWAP ? sfy : sfx;
#pragma unroll
      for (int a = 0; a < C::ACT_ATOMS; ++a)
        *reinterpret_cast<uint4*>(act_sf + a * kSfAtomBytes + lane * 16) =
            make_uint4(words[4 * a], words[4 * a + 1], words[4 * a + 2], words[4 * a + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&full[s]);
      ++issued;
      if (it + 1 < nk) gather(kg + 1);
    }
    // Drain: every issued stage's copies must have landed before exit.
    for (int it = max(0, issued - NSTAGE); it < issued; ++it) {
      if (!ptx::mbar_wait(&full[it % NSTAGE], (uint32_t)(it / NSTAGE) & 1u, kWaitLimitNs)) {
        watchdog(abort_flag, kWdDrain);
        break;
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    for (int it = 0; it < nk; ++it) {
      const int s = it % NSTAGE;
      const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
      if (*abort_flag) break;
      if (!ptx::mbar_wait(&full[s], ph, kWaitLimitNs)) {
        watchdog(abort_flag, kWdMma);
        break;
      }
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint32_t sfx_col = tmem + BN + s * C::SF_COLS;
        const uint32_t sfy_col = sfx_col + 4;
        const uint32_t xs = ptx::smem_u32(smem + C::OFF_X + s * C::X_TILE);
        const uint32_t ys = ptx::smem_u32(smem + C::OFF_Y + s * C::Y_TILE);
        const uint32_t sfx = ptx::smem_u32(smem + C::OFF_SFX + s * C::SFX_BYTES);
        const uint32_t sfy = ptx::smem_u32(smem + C::OFF_SFY + s * C::SFY_BYTES);
        ptx::tmem_cp_32x128b_x4(sfx_col, ptx::smem_desc(sfx, 128, 128, ptx::kSwizzleNone));
#pragma unroll
        for (int a = 0; a < C::Y_ATOMS; ++a)
          ptx::tmem_cp_32x128b_x4(sfy_col + 4 * a, ptx::smem_desc(sfy + a * kSfAtomBytes, 128, 128,
                                                                  ptx::kSwizzleNone));
        const uint64_t adesc = ptx::smem_desc(xs, 16, 1024, ptx::kSwizzle128B);
        const uint64_t bdesc = ptx::smem_desc(ys, 16, 1024, ptx::kSwizzle128B);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // 4 x (K = 32 bytes) inside the 128-byte swizzle row
          ptx::mma_mxf8(tmem, adesc + 2 * k, bdesc + 2 * k, C::IDESC, sfx_col, sfy_col,
                        (it > 0 || k > 0) ? 1u : 0u);
        ptx::tc_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (lane == 0) ptx::tc_commit(acc_full);  // also after an abort: tracks what was issued
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;
    const bool waited = ptx::mbar_wait(acc_full, 0, kWaitLimitNs);
    if (!waited) watchdog(abort_flag, kWdEpilogue);
    ptx::tc_fence_after();
    const bool ok = __all_sync(0xffffffffu, waited) && !*abort_flag;
    if (ok) {
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
      float* part = reinterpret_cast<float*>(smem);  // stage buffers are idle now
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t v[16];
        ptx::tmem_ld_32x32b_x16(trow + c * 16, v);
        ptx::tmem_ld_wait();
        if (nk == 0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0u;  // empty K slice contributes zero
        }
        if (!SWAP) {
          const int t = x0 + r;
          const int n = y0 + c * 16;
          if (t < p.T && n < p.N) {
            uint4 lo, hi;
            lo.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
            lo.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
            lo.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
            lo.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
            hi.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
            hi.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
            hi.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
            hi.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((size_t)t * p.G + g) * p.N + n);
            dst[0] = lo;
            dst[1] = hi;
          }
        } else if (p.splits == 1) {
          const int n = x0 + r;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = y0 + c * 16 + j;
            if (t < p.T && n < p.N)
              p.out[((size_t)t * p.G + g) * p.N + n] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) part[r * C::PART_PITCH + c * 16 + j] = __uint_as_float(v[j]);
        }
      }
    }
    ptx::tc_fence_before();
  }

  __syncthreads();
  if (SWAP && p.splits > 1) {
    // Deterministic split-K reduction over the cluster: CTA `split` sums
    // rows [split*rows, (split+1)*rows) of the tile over ranks 0..splits-1.
    ptx::cluster_sync();
    const int rows = (C::BM + p.splits - 1) / p.splits;
    const int r_begin = split * rows;
    const int r_end = min(C::BM, r_begin + rows);
    const int tv = min(BN, p.T - y0);
    const int nrows = r_end - r_begin;
    if (!*abort_flag && nrows > 0 && tv > 0) {
      const uint32_t part0 = ptx::smem_u32(smem);
      for (int e = threadIdx.x; e < nrows * tv; e += kThreads) {
        const int tl = e / nrows;
        const int rr = r_begin + e % nrows;
        const uint32_t off = (uint32_t)(rr * C::PART_PITCH + tl) * 4u;
        float acc = 0.0f;
        for (int rk = 0; rk < p.splits; ++rk)
          acc += ptx::ld_shared_cluster_f32(ptx::map_shared_rank(part0 + off, (uint32_t)rk));
        const int n = x0 + rr;
        if (n < p.N) p.out[((size_t)(y0 + tl) * p.G + g) * p.N + n] = __float2bfloat16_rn(acc);
      }
    }
    ptx::cluster_sync();  // keep every partial tile alive until all readers are done
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// --------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D uint8 tensor map, inner dimension K with 128-byte rows swizzled, zero
// fill outside the tensor.
bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool SWAP, int BN, int NSTAGE>
cudaError_t launch_cfg(const uint8_t* a, const uint8_t* w, BmmArgs args, cudaStream_t s,
                       const char** why) {
  using C = Cfg<SWAP, BN, NSTAGE>;
  const uint64_t K = args.K, G = args.G, T = args.T, N = args.N;
  CUtensorMap tm_act, tm_w;
  const uint32_t act_box = SWAP ? BN : C::BM;
  const uint32_t w_box = SWAP ? C::BM : BN;
  if (!encode_3d(&tm_act, a, K, G, T, K, G * K, 128, 1, act_box) ||
      !encode_3d(&tm_w, w, K, N, G, K, N * K, 128, w_box, 1)) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point missing or arguments rejected)";
    return cudaErrorInvalidValue;
  }
  auto kern = bmm_a8w8_kernel<SWAP, BN, NSTAGE>;
  // The shared-memory opt-in is set once per device (a host-side call that
  // must not run inside stream capture, so the first call on a device should
  // happen before any capture).
  static std::atomic<uint64_t> smem_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(smem_set.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    smem_set.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(args.x_tiles * args.y_tiles * args.splits), (unsigned)args.G, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (args.splits > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)args.splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, tm_act, tm_w, args);
}

}  // namespace

cudaError_t launch_bmm_a8w8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* w,
                            const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                            int num_sms, cudaStream_t s, const char** why) {
  BmmArgs args;
  args.a_sf = a_sf;
  args.w_sf = w_sf;
  args.out = reinterpret_cast<__nv_bfloat16*>(out);
  args.T = (int)T;
  args.G = G;
  args.N = N;
  args.K = K;
  args.KG = (int)ceil_div(K, kGroup);
  args.NB = (int)sf_row_blocks(N);
  if (T <= 128) {
    // Few tokens: weight rows on the MMA M axis, tokens on N.
    const int bn = T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128;
    args.x_tiles = (int)ceil_div(N, 128);
    args.y_tiles = 1;
    const int base = args.x_tiles * G;
    int splits = num_sms / (base > 0 ? base : 1);
    splits = splits < 1 ? 1 : (splits > 8 ? 8 : splits);
    splits = splits > args.KG ? args.KG : splits;
    args.kg_per_split = (int)ceil_div(args.KG, splits);
    args.splits = (int)ceil_div(args.KG, args.kg_per_split);
    switch (bn) {
      case 16: return launch_cfg<true, 16, 10>(a, w, args, s, why);
      case 32: return launch_cfg<true, 32, 10>(a, w, args, s, why);
      case 64: return launch_cfg<true, 64, 8>(a, w, args, s, why);
      default: return launch_cfg<true, 128, 6>(a, w, args, s, why);
    }
  }
  args.x_tiles = (int)ceil_div(T, 128);
  args.y_tiles = (int)ceil_div(N, 256);
  args.splits = 1;
  args.kg_per_split = args.KG;
  return launch_cfg<false, 256, 4>(a, w, args, s, why);
}

cudaError_t watchdog_read(uint32_t* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_watchdog, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_watchdog, &zero, sizeof(uint32_t));
  }
  return e;
}

}  // namespace mxq
