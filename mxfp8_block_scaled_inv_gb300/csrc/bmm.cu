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
// Work unit = one output tile of one group g (and, for the split-K form, one
// K slice of it).  Warp roles (12 warps; 11 in the fused form; the pair
// form adds a gate warp 12 that waits on the MMA warp's barriers, and the
// quantising pair form, which has no scale loader, runs that gate on warp
// 2):
//   warp 0      weight producer: per pipeline stage (one 128-wide K group) a
//               TMA load of the W tile (128-byte swizzle, zero fill outside
//               the tensor: this is the unaligned-K tail) and a copy of the
//               prepared weight-scale atom(s).
//   warp 1      TMEM owner and MMA issuer: per stage, tcgen05.cp of the scale
//               atoms into TMEM, four tcgen05.mma kind::mxf8f6f4 block_scale
//               (K = 32 each; every word of an atom holds its group's byte four
//               times, so each 32-block sees the group scale), tcgen05.commit
//               to free the stage; per tile a commit that hands the fp32
//               accumulator to the epilogue.
//   warp 2      activation-scale loader: copies the tile's scale bytes (one
//               row per token, up to 64 groups at a time) from global memory
//               into a double-buffered compact buffer ahead of the producers.
//   warps 3-10  epilogue: two warps per TMEM lane quadrant, each draining half
//               of the tile's columns into registers, then releasing the
//               accumulator to the MMA warp before rounding to BF16 and
//               storing, so the next tile's MMAs overlap the stores.
//   warp 11     activation producer: per stage the TMA load of the activation
//               tile and the stage's activation-scale atom, built from the
//               compact buffer.  Weights and activations come from two warps
//               because one thread completes only about one TMA copy every
//               ~540 cycles.
// Three forms:
//   pair    (many tokens): a cluster of two CTAs issues the 2-SM MMA
//           (tcgen05 cta_group::2): M = 256 tokens, 128 per CTA, N = 256
//           weight rows, of which each CTA loads 128 while holding the scale
//           atoms of all 256.  The CTA pairs are persistent and walk the
//           units with the weight tile fastest, so concurrent pairs share A
//           and W tiles through L2.
//   swapped (few tokens):  MMA M = 128 weight rows, MMA N = 16..128 tokens, so
//           the weight streams at full tile width with no padding of the token
//           axis to 128.  The K range may be split over the CTAs of a
//           thread-block cluster, whose fp32 partial tiles are summed in rank
//           order through distributed shared memory (deterministic, no global
//           workspace).
//   fused   (swapped, T <= 32): the activation is read as BF16 straight from
//           the attention output by TMA, and the epilogue warps, idle during
//           the mainloop, quantise each stage's tokens (inverse RoPE on the
//           last group, group-128 E8M0 scale, E4M3 codes) directly into the
//           128-byte-swizzled operand tile and the scale atom the MMA reads.
//           One launch then does the whole wo_a (or MXFP8 linear) step, with
//           no round trip of the codes through HBM.
//   pair + quantise (many tokens, wo_a): the pair form, reading the BF16
//           activation.  Between accumulator drains the 8 epilogue warps
//           quantise the CTA's own 128 token rows (inverse RoPE on the last
//           group, group scale, E4M3 codes) into a workspace, independently
//           of the MMAs: the codes go to global memory in the [T][G][K]
//           layout and the scale bytes as ready-made scale atoms, and a
//           per-(128 rows, K group) counter in global memory is raised once
//           the writes are visible.  The units of one 256-token block are
//           taken by consecutive pairs, and the y_tiles pairs that share it
//           split its K groups, so the quantisation is spread over every SM
//           and done once.  The activation producer reads the counters and
//           TMA-loads the codes and atoms as soon as they are published.  The
//           quantising work waits only for its own copies, so the counters
//           always complete (every CTA of the persistent grid is resident).
//           This form has no scale loader: its gate runs on warp 2 and the
//           CTA has 12 warps, which leaves 168 registers per thread (three
//           warps per SM sub-partition instead of four).
// Every wait is bounded in wall time; on expiry the kernel sets a watchdog
// bit, stops issuing, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>
#include <utility>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"
#include "mxq_ptx.cuh"
#include "quant_common.cuh"

namespace mxq {

__device__ uint32_t g_watchdog;
// Jobs of the one-launch prefill quantised by a consumer (a testing aid).
__device__ uint32_t g_takeovers;

// Cap on the CTA pairs of the pair forms (0: one pair per co-resident
// cluster slot); a testing aid, see mxq_debug_set_pair_limit.
std::atomic<int> g_pair_limit{0};
// Testing aid, see mxq_debug_set_lazy_pairs: pairs from this index on skip
// their quantisation jobs (as if they never started).
std::atomic<int> g_lazy_from{1 << 30};

namespace {

constexpr uint64_t kWaitLimitNs = 4000000000ull;
// Longest a pipeline wait may sleep before re-checking: stages turn over
// every few hundred nanoseconds, and a plain try_wait measured up to ~1.6 us
// late in waking after its phase completed.
constexpr uint32_t kPipeHintNs = 20;
constexpr uint32_t kWdProducer = 1, kWdMma = 2, kWdEpilogue = 4, kWdDrain = 8, kWdLoader = 16;
constexpr int kEpiWarp0 = 3;   // epilogue warps 3-10
constexpr int kEpiWarps = 8;
constexpr int kActWarp = 11;   // activation producer (unfused forms)
constexpr int kGateWarp = 12;  // pair form: waits on the MMA warp's barriers
constexpr int kQGateWarp = 2;  // the same role in the quantising pair form
// Quantising pair form: a job (128 rows of one K group) is kQSlices slices
// of 16 rows x 128 values, and epilogue warp w quantises slice w of every
// job of its CTA, between accumulator drains, from its own shared-memory slot
// that it refills itself with TMA; a job's counter reaches kQSlices.
constexpr int kQWorkers = kEpiWarps;
constexpr int kQSlices = 8;
constexpr int kQRows = 128 / kQSlices;
constexpr int kQSliceBytes = kQRows * 128 * 2;
constexpr int kQSlots = kQWorkers;
static_assert(kQSlices == kQWorkers, "one slice of every job per epilogue warp");
// Longest sleep between two polls of a not-yet-published counter, and
// between two polls of an epilogue warp with nothing ready.
constexpr uint32_t kFlagPollNs = 128;
constexpr uint32_t kEpiPollNs = 32;
// Each quantising warp prefetches its slice of the job this many jobs ahead
// into L2 (its shared-memory copies then wait on L2, not DRAM).
constexpr int kQPrefetch = 2;
// Quantisation runs at most this many units ahead of the CTA's GEMM.
constexpr int kQLead = 1;
// Publications are batched (and made at once whenever the warp has nothing
// else ready): the gpu-scope fence waits for every store the warp still has
// in flight.
constexpr int kQPublish = 4;
// A job that a consumer has waited on this long is quantised by the
// consumer itself (its owner may not be running, e.g. while a kernel of
// another stream holds SMs); in normal operation no wait comes near it.
constexpr uint64_t kTakeoverNs = 50000;

struct BmmArgs {
  const uint8_t* a_sf;  // [T][G][KG]
  const uint8_t* w_sf;  // prepared: [G][KG][NB][512]
  __nv_bfloat16* out;   // [T][G][N]
  int T, G, N, K, KG, NB;
  int x_tiles, y_tiles;  // tiles along the MMA-A rows (128) and MMA-B rows (BN)
  int splits, kg_per_split;
  int x_span;            // rows of the MMA-A side per unit (256 for a CTA pair)
  int units;             // G * x_tiles * y_tiles * splits
  int persistent;        // 1: each CTA (pair) walks units with stride = CTAs (pairs) in the grid
  // Fused activation form only: positions, cos/sin cache, RoPE width.
  const int64_t* pos;
  const uint16_t* cos_tab;
  const uint16_t* sin_tab;
  int64_t cs_ld, max_pos;
  int R;
  int32_t* err_flag;
  // Quantising pair form only: BF16 input and the workspace it fills.
  const uint16_t* xq;  // [T][G][K] BF16
  uint8_t* qcodes;     // [T][G][K] E4M3 codes (read back as the A operand)
  uint8_t* qatoms;     // [G][MB][KG][512] activation scale atoms
  uint32_t* qflags;    // [G][MB][KG] job counters, zero before the launch
  int MB;              // 128-token blocks per group (2 * x_tiles)
  int q_lazy_from;     // testing aid: pairs from this index on quantise nothing
};

// PAIR: the CTA-pair form (normal orientation only): MMA M = 256 tokens, 128
// per CTA; MMA N = BN weight rows, of which each CTA loads half, while each
// holds the scale atoms of all BN rows.  QUANT (pair form only): the kernel
// quantises the BF16 activation itself.
template <bool SWAP, bool FUSED, int BN, int NSTAGE, bool PAIR = false, bool QUANT = false>
struct Cfg {
  static constexpr int BM = 128;
  static constexpr int BK = 128;
  static constexpr int Y_ATOMS = (BN + 127) / 128;
  static constexpr int ACT_ROWS = SWAP ? BN : BM;
  static constexpr int X_TILE = BM * BK;
  static constexpr int Y_ROWS = PAIR ? BN / 2 : BN;  // MMA-B rows held by this CTA
  static constexpr int Y_TILE = Y_ROWS * BK;
  static constexpr int SFX_BYTES = kSfAtomBytes;
  static constexpr int SFY_BYTES = Y_ATOMS * kSfAtomBytes;
  static constexpr int W_SF_BYTES = (SWAP ? 1 : Y_ATOMS) * kSfAtomBytes;
  // Compact activation-scale buffer: groups per chunk (a few-token CTA holds
  // only a short K slice; the pair form spends the shared memory on a sixth
  // pipeline stage instead).
  static constexpr int SF_CHUNK = (SWAP || PAIR) ? 16 : 64;
  static constexpr int CSF_BYTES = (FUSED || QUANT) ? 0 : SF_CHUNK * 128;  // [group][128 rows]
  static constexpr int STG_BYTES = FUSED ? BN * 256 : 0;         // BF16 staging [BN][128]
  static constexpr int OFF_X = 0;
  static constexpr int OFF_Y = OFF_X + NSTAGE * X_TILE;
  static constexpr int OFF_SFX = OFF_Y + NSTAGE * Y_TILE;
  static constexpr int OFF_SFY = OFF_SFX + NSTAGE * SFX_BYTES;
  static constexpr int OFF_STG = OFF_SFY + NSTAGE * SFY_BYTES;
  static constexpr int OFF_CSF = OFF_STG + NSTAGE * STG_BYTES;
  // fp32 split-K receive buffer of the swapped form: [split][rows owned][BN+4]
  // with rows owned = ceil(128 / splits); splits * that <= 133 for splits <= 8.
  static constexpr int PART_PITCH = BN + 4;
  static constexpr int RED_ROWS = 136;
  static constexpr int RED_BYTES = SWAP ? RED_ROWS * PART_PITCH * 4 : 0;
  static constexpr int OFF_RED = OFF_CSF + 2 * CSF_BYTES;
  // Pair form: per epilogue warp, one 32 x 32 BF16 staging tile for the
  // TMA stores of the output.
  static constexpr int OUT_TILE = 32 * 32 * 2;
  static constexpr int OUT_BYTES = PAIR ? 8 * OUT_TILE : 0;
  static constexpr int OFF_OUT = OFF_RED + RED_BYTES;
  // Quantising form: the BF16 activation slices.
  static constexpr int QX_BYTES = QUANT ? kQSlots * kQSliceBytes : 0;
  static constexpr int OFF_QX = OFF_OUT + OUT_BYTES;
  // Quantising form: the activation producer's slot for quantising a job
  // whose owner is late (one slice at a time).
  static constexpr int TK_BYTES = QUANT ? kQSliceBytes : 0;
  static constexpr int OFF_TK = OFF_QX + QX_BYTES;
  static constexpr int OFF_BAR = OFF_TK + TK_BYTES;
  // full[NSTAGE], empty[NSTAGE], landed[NSTAGE], acc_full, acc_empty,
  // sf_full[2], sf_empty[2], mma_done, then qfull[kQSlots] and the takeover
  // slot's barrier
  static constexpr int N_BARS = 3 * NSTAGE + 7 + (QUANT ? kQSlots + 1 : 0);
  static constexpr int OFF_SLOT = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_SLOT + 16 + 1024;
  // Two CTAs share an SM when their shared memory allows it (the small-token
  // forms): more K slices stream at once, and with programmatic dependent
  // launch the next call's CTAs start streaming weights beside this one's.
  static constexpr int CTAS_PER_SM = SMEM_BYTES <= 113 * 1024 ? 2 : 1;
  static constexpr int SF_COLS = 4 + 4 * Y_ATOMS;
  static constexpr int TMEM_USED = BN + NSTAGE * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                   : TMEM_USED <= 64  ? 64
                                   : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256
                                                      : 512;
  static constexpr int HALF = BN / 2;        // columns drained by one epilogue warp
  // The fused form quantises in the epilogue warps and needs no activation
  // producer warp.
  // The pair form adds a gate warp that does the MMA warp's barrier waits:
  // the tensor pipe's instruction queue is shallow, so any wait in the
  // issuing warp between stages leaves the pipe idle.  The quantising pair
  // form needs no scale loader and runs its gate on that warp.
  static constexpr int THREADS = (FUSED ? 11 : (PAIR && !QUANT ? 13 : 12)) * 32;
  // Instruction descriptor, kind::mxf8f6f4 with block scaling: E4M3 A and
  // B (format 0), both K-major, N >> 3 at bits 17-22, UE8M0 scale type at
  // bit 23, M >> 4 at bits 24-28, scale-factor ids 0.
  static constexpr uint32_t IDESC =
      (1u << 23) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((PAIR ? 2 * BM : BM) >> 4) << 24);
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(!FUSED || (SWAP && BN <= 32), "fused activations: swapped form, <= 32 tokens");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
  static_assert(ACT_ROWS <= 128, "activation scale rows fit one loader pass");
  static_assert(HALF % 8 == 0, "epilogue drains 8-column chunks");
  static_assert(!PAIR || (!SWAP && !FUSED && BN == 256), "pair form: normal orientation, N = 256");
  static_assert(!QUANT || PAIR, "in-kernel quantisation: pair form only");
};

__device__ __forceinline__ void watchdog(volatile int* abort_flag, uint32_t bit) {
  *abort_flag = 1;
  atomicOr(&g_watchdog, bit);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 r = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Decoded work unit.  The weight tile index runs fastest.
struct Unit {
  int g, x0, y0, split, kg_begin, nk;
};

template <bool SWAP, int BN>
__device__ __forceinline__ Unit decode_unit(const BmmArgs& p, int u) {
  Unit w;
  w.split = u % p.splits;
  int r = u / p.splits;
  int xt, yt;
  if (!SWAP) {  // weights on Y
    yt = r % p.y_tiles;
    r /= p.y_tiles;
    xt = r % p.x_tiles;
    r /= p.x_tiles;
  } else {  // weights on X
    xt = r % p.x_tiles;
    r /= p.x_tiles;
    yt = r % p.y_tiles;
    r /= p.y_tiles;
  }
  w.g = r;
  w.x0 = xt * p.x_span;
  w.y0 = yt * BN;
  w.kg_begin = w.split * p.kg_per_split;
  w.nk = max(0, min(p.KG, w.kg_begin + p.kg_per_split) - w.kg_begin);
  return w;
}

// ------------------------------------------- in-kernel activation quantisation
// A job = one K group kg of one 128-token block of one group g, done by the
// CTA that owns the block as kQSlices slices of kQRows rows, slice w by
// epilogue warp w from its own shared-memory slot; each slice raises the
// job's counter by one, so a finished job's counter reads kQSlices.
struct QJob {
  int u, jj;  // unit and job index within the unit
  int g, kg;  // group and K group
  int t0;     // first token of the 128-token block
  int f;      // counter / atom index: (g * MB + block) * KG + kg
};

// Job jj of unit u for CTA `rank` of the pair: of the y_tiles pairs that
// share a 256-token block, the one holding weight tile yt quantises K groups
// r, r + y_tiles, ... with r = (yt + block) mod y_tiles, so that the rotated
// last group (the slowest) moves from pair to pair with the block.
__device__ __forceinline__ bool qjob_make(const BmmArgs& p, int u, int jj, int rank, QJob& j) {
  const Unit w = decode_unit<false, 256>(p, u);
  const int kg = (w.y0 / 256 + w.x0 / 256) % p.y_tiles + jj * p.y_tiles;
  if (kg >= p.KG) return false;
  const int blk = w.x0 / 128 + rank;
  j.u = u;
  j.jj = jj;
  j.g = w.g;
  j.kg = kg;
  j.t0 = blk * 128;
  j.f = (w.g * p.MB + blk) * p.KG + kg;
  return true;
}

// Advances j to the next job of this CTA (units u, u + u_step, ...).
__device__ __forceinline__ bool qjob_next(const BmmArgs& p, int u_step, int rank, QJob& j) {
  if (j.kg + p.y_tiles < p.KG) {  // the same unit's next K group
    ++j.jj;
    j.kg += p.y_tiles;
    j.f += p.y_tiles;
    return true;
  }
  for (int u = j.u + u_step; u < p.units; u += u_step)
    if (qjob_make(p, u, 0, rank, j)) return true;
  return false;
}

__device__ __forceinline__ bool qjob_first(const BmmArgs& p, int u_first, int u_step, int rank,
                                           QJob& j) {
  for (int u = u_first; u < p.units; u += u_step)
    if (qjob_make(p, u, 0, rank, j)) return true;
  return false;
}

// Quantises a rotated slice (the row's last group when R > 0; one in KG
// jobs): steps of two rows, a half-warp per row and 8 values per lane, with
// the arithmetic of the standalone quantiser: inverse rotation (lower lanes
// fetch cos, their partners sin, for the same indices), group abs-max,
// scale, codes.  The cos/sin operands of all 8 steps are fetched first (one
// round trip), then the values, then the steps run unrolled.  Codes go to
// [T][G][K]; the scale of row r = 16 s + rr of the block goes to atom line
// r % 32, word r / 32 (rows past T: 127; invalid position: zero codes,
// scale 0).
__device__ __forceinline__ void qslice_rope(const BmmArgs& p, const QJob& j, int s,
                                            const uint8_t* buf, int lane, uint32_t badmask,
                                            int64_t pl) {
  const int hw = lane >> 4;
  const int sub = lane & 15;
  const int c = j.kg * 16 + sub;
  const int t0 = j.t0 + kQRows * s;
  const int first = 16 - (p.R >> 3);
  const int dist = p.R >> 4;
  const bool rope_lane = sub >= first;
  const bool lower = sub < first + dist;
  const int partner = (hw << 4) | (rope_lane ? (lower ? sub + dist : sub - dist) : sub);
  const int i0 = (sub - first - (lower ? 0 : dist)) * 8;
  const uint16_t* tab = lower ? p.cos_tab : p.sin_tab;
  uint8_t* arow = p.qatoms + (size_t)j.f * kSfAtomBytes + (16 * (s & 1)) * 16 + (s >> 1) * 4;
  uint4 cs[kQRows / 2];
#pragma unroll
  for (int i = 0; i < kQRows / 2; ++i) {
    const int rr = 2 * i + hw;
    const int64_t pp = __shfl_sync(0xffffffffu, (long long)pl, rr);
    const bool rot = rope_lane && !((badmask >> rr) & 1u) && t0 + rr < p.T;
    cs[i] = make_uint4(0, 0, 0, 0);
    if (rot) cs[i] = __ldg(reinterpret_cast<const uint4*>(tab + pp * p.cs_ld + i0));
  }
  uint4 v[kQRows / 2];
#pragma unroll
  for (int i = 0; i < kQRows / 2; ++i)
    v[i] = *reinterpret_cast<const uint4*>(buf + (2 * i + hw) * 256 + sub * 16);
#pragma unroll
  for (int i = 0; i < kQRows / 2; ++i) {
    const int rr = 2 * i + hw;
    const int t = t0 + rr;
    const bool bad = (badmask >> rr) & 1u;
    uint4 o, pv;
    o.x = __shfl_sync(0xffffffffu, cs[i].x, partner);
    o.y = __shfl_sync(0xffffffffu, cs[i].y, partner);
    o.z = __shfl_sync(0xffffffffu, cs[i].z, partner);
    o.w = __shfl_sync(0xffffffffu, cs[i].w, partner);
    pv.x = __shfl_sync(0xffffffffu, v[i].x, partner);
    pv.y = __shfl_sync(0xffffffffu, v[i].y, partner);
    pv.z = __shfl_sync(0xffffffffu, v[i].z, partner);
    pv.w = __shfl_sync(0xffffffffu, v[i].w, partner);
    float y[8];
    unpack8(v[i], y);
    if (rope_lane && !bad && t < p.T) {
      float xp[8];
      unpack8(pv, xp);
      inv_rope8(y, xp, lower ? cs[i] : o, lower ? o : cs[i], lower);
    }
    uint32_t sb;
    uint2 q8 = encode8(y, half_warp_amax(y), &sb);
    q8 = bad ? make_uint2(0, 0) : q8;
    sb = bad ? 0u : sb;
    if (c * 8 < p.K && t < p.T)
      *reinterpret_cast<uint2*>(p.qcodes + ((size_t)t * p.G + j.g) * p.K + c * 8) = q8;
    if (sub == 0) *reinterpret_cast<uint32_t*>(arow + rr * 16) = (t < p.T ? sb : 127u) * 0x01010101u;
  }
}

// Quantises a plain slice from its slot: 8 lanes per row, 16 values per
// lane (elements [8 l, 8 l + 8) and [64 + 8 l, 64 + 8 l + 8) of the row's
// group for lane l of the row's 8, so each shared-memory read is 128
// contiguous bytes per row), four rows per step.  The values of all four
// steps are read into registers and the slot is released (`release`), then
// the abs-max of every step is taken (the shuffle trees interleave), then
// every step's scale and codes, then `before_stores` runs and the codes and
// atom words are stored, with the same arithmetic as the standalone
// quantiser.  Rows past T: no codes, scale 127; rows with an invalid
// position: zero codes, scale 0; row r = 16 s + 4 i + r4 of the block sits
// at atom line r % 32, word r / 32.
template <class Release, class BeforeStores>
__device__ __forceinline__ void qslice_plain(const BmmArgs& p, const QJob& j, int s,
                                             const uint8_t* buf, int lane, uint32_t badmask,
                                             Release&& release, BeforeStores&& before_stores) {
  const int r4 = lane >> 3;  // row of the step
  const int l8 = lane & 7;   // the row's lane
  const int t0 = j.t0 + kQRows * s;
  uint4 va[4], vb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t* row = buf + (4 * i + r4) * 256 + l8 * 16;
    va[i] = *reinterpret_cast<const uint4*>(row);
    vb[i] = *reinterpret_cast<const uint4*>(row + 128);
  }
  release();
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float ya[8], yb[8];
    unpack8(va[i], ya);
    unpack8(vb[i], yb);
    float mx = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fmaxf(fabsf(ya[e]), fabsf(yb[e])));
    m[i] = mx;
  }
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], d));
  uint2 qa[4], qb[4];
  uint32_t sw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float ya[8], yb[8];
    unpack8(va[i], ya);
    unpack8(vb[i], yb);
    uint32_t sb;
    qa[i] = encode8(ya, m[i], &sb);
    qb[i] = encode8(yb, m[i], &sb);
    const int rr = 4 * i + r4;
    const bool bad = (badmask >> rr) & 1u;
    qa[i] = bad ? make_uint2(0, 0) : qa[i];
    qb[i] = bad ? make_uint2(0, 0) : qb[i];
    sw[i] = (t0 + rr < p.T ? (bad ? 0u : sb) : 127u) * 0x01010101u;
  }
  before_stores();
  const int ca = j.kg * 128 + l8 * 8;
  uint8_t* crow = p.qcodes + ((size_t)(t0 + r4) * p.G + j.g) * p.K + ca;
  const size_t cstep = (size_t)4 * p.G * p.K;
  uint8_t* arow = p.qatoms + (size_t)j.f * kSfAtomBytes + (16 * (s & 1) + r4) * 16 + (s >> 1) * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (t0 + 4 * i + r4 < p.T) {
      if (ca < p.K) *reinterpret_cast<uint2*>(crow + i * cstep) = qa[i];
      if (ca + 64 < p.K) *reinterpret_cast<uint2*>(crow + i * cstep + 64) = qb[i];
    }
    if (l8 == 0) *reinterpret_cast<uint32_t*>(arow + i * 64) = sw[i];
  }
}

// Quantises job (g, 128-token block starting at t0, K group kg), counter f,
// in the calling warp, one 16-row slice at a time through the warp's own
// slot `tslot` (barrier `tbar`, whose phase bit `tphase` it advances), and
// raises the counter by kQSlices.  Used by a consumer whose wait on the
// job's owner ran long.  Lane r < 16 does row r of each slice on its own, in
// two passes over the slot (group abs-max, then codes), with the helpers and
// the order of operations of the epilogue warps, so the bytes are the same;
// the owner may still quantise the same job (both write the same bytes, and
// a counter above kQSlices reads as complete).  Written for few live
// registers: it sits in the kernel's rarely taken path, and a larger
// footprint there would cost the whole kernel registers.  Returns false when
// a copy did not land in time.
__device__ __forceinline__ bool take_over_job(const BmmArgs& p, const CUtensorMap* xq,
                                              uint8_t* tslot, uint64_t* tbar, uint32_t& tphase,
                                              int g, int kg, int t0, int f, int lane) {
  const bool rope = p.R > 0 && kg == p.KG - 1;
  const int first = 16 - (p.R >> 3);  // first chunk of the rotated slice
  const int dist = p.R >> 4;          // chunks between rotate-half partners
  for (int sl = 0; sl < kQSlices; ++sl) {
    ptx::fence_proxy_async_smem();  // the slot's previous contents were read
    __syncwarp();
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(tbar, kQSliceBytes);
      ptx::tma_load_3d(tslot, xq, tbar, kg * 128, g, t0 + kQRows * sl);
    }
    const bool landed_ok = ptx::mbar_wait(tbar, tphase, kWaitLimitNs);
    tphase ^= 1u;
    if (!__all_sync(0xffffffffu, landed_ok)) return false;
    if (lane < kQRows) {
      const int rr = kQRows * sl + lane;  // row within the 128-token block
      const int t = t0 + rr;
      const bool valid = t < p.T;
      const int64_t pl = (p.R > 0 && valid) ? __ldg(p.pos + t) : 0;
      const bool bad = p.R > 0 && valid && (pl < 0 || pl >= p.max_pos);
      const uint8_t* row = tslot + lane * 256;
      // The fp32 values of chunk c (8 elements), rotated when c lies in the
      // slice: inverse RoPE against the partner chunk R/16 chunks away, with
      // the cos/sin entries both halves of a pair share.
      auto chunk = [&](int c, float (&y)[8]) {
        unpack8(*reinterpret_cast<const uint4*>(row + c * 16), y);
        if (rope && c >= first && valid && !bad) {
          const bool lower = c < first + dist;
          float xp[8];
          unpack8(*reinterpret_cast<const uint4*>(row + (lower ? c + dist : c - dist) * 16), xp);
          const int i0 = (c - first - (lower ? 0 : dist)) * 8;
          const uint4 cw = __ldg(reinterpret_cast<const uint4*>(p.cos_tab + pl * p.cs_ld + i0));
          const uint4 sw = __ldg(reinterpret_cast<const uint4*>(p.sin_tab + pl * p.cs_ld + i0));
          inv_rope8(y, xp, cw, sw, lower);
        }
      };
      float amax = 0.0f;
      for (int c = 0; c < 16; ++c) {
        float y[8];
        chunk(c, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(y[e]));
      }
      uint32_t sb = 0;
      for (int c = 0; c < 16; ++c) {
        float y[8];
        chunk(c, y);
        uint2 q8 = encode8(y, amax, &sb);
        if (bad) q8 = make_uint2(0, 0);
        const int col = kg * 128 + c * 8;
        if (valid && col < p.K)
          *reinterpret_cast<uint2*>(p.qcodes + ((size_t)t * p.G + g) * p.K + col) = q8;
      }
      *reinterpret_cast<uint32_t*>(p.qatoms + (size_t)f * kSfAtomBytes + (rr % 32) * 16 +
                                   (rr / 32) * 4) = (valid ? (bad ? 0u : sb) : 127u) * 0x01010101u;
      if (bad && kg == 0 && p.err_flag != nullptr) atomicOr(p.err_flag, MXQ_DEVERR_POSITION);
    }
  }
  // Publish as the epilogue warps do: the codes and atom words are read by
  // other CTAs through TMA.
  ptx::fence_proxy_async_global();
  ptx::fence_acq_rel_gpu();
  __syncwarp();
  if (lane == 0) ptx::red_add_relaxed_gpu(p.qflags + f, (uint32_t)kQSlices);
  return true;
}

// Tensor maps only the quantising form takes (the activation scale atoms it
// writes and its BF16 input); the other forms take an empty parameter, so
// that their launches copy no more parameter bytes than they use.
struct QuantMaps {
  CUtensorMap asf, xq;
};
struct NoMaps {};
template <bool QUANT>
using QuantMapsT = typename std::conditional<QUANT, QuantMaps, NoMaps>::type;
__device__ __forceinline__ const CUtensorMap* map_asf(const QuantMaps& m) { return &m.asf; }
__device__ __forceinline__ const CUtensorMap* map_xq(const QuantMaps& m) { return &m.xq; }
__device__ __forceinline__ const CUtensorMap* map_asf(const NoMaps&) { return nullptr; }
__device__ __forceinline__ const CUtensorMap* map_xq(const NoMaps&) { return nullptr; }

template <bool SWAP, bool FUSED, int BN, int NSTAGE, bool PAIR, bool QUANT>
__global__ void __launch_bounds__((Cfg<SWAP, FUSED, BN, NSTAGE, PAIR, QUANT>::THREADS),
                                  (Cfg<SWAP, FUSED, BN, NSTAGE, PAIR, QUANT>::CTAS_PER_SM))
    bmm_a8w8_kernel(const __grid_constant__ CUtensorMap tm_act,
                    const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ CUtensorMap tm_wsf,
                    const __grid_constant__ CUtensorMap tm_out,
                    const __grid_constant__ QuantMapsT<QUANT> qmaps, const BmmArgs p) {
  using C = Cfg<SWAP, FUSED, BN, NSTAGE, PAIR, QUANT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NSTAGE;
  uint64_t* landed = empty + NSTAGE;  // fused form: a stage's copies have landed
  uint64_t* acc_full = landed + NSTAGE;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* sf_full = acc_empty + 1;
  uint64_t* sf_empty = sf_full + 2;
  uint64_t* mma_done = sf_empty + 2;
  uint64_t* qfull = mma_done + 1;  // quantising form only: the epilogue warps' slots
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SLOT);
  uint8_t* csf = smem + C::OFF_CSF;
  __shared__ int abort_shared;
  __shared__ int act_done_shared;  // stages the activation producer completed
  __shared__ int gate_go_shared[2];  // pair form: stage handed over (1) or stop (0)
  volatile int* abort_flag = &abort_shared;
  volatile int* act_done = &act_done_shared;
  volatile int* gate_go = gate_go_shared;

  // The next kernel on the stream may be scheduled from the start: it only
  // streams its own weights until it has waited for this grid to complete.
  // (Triggered here rather than after this CTA's set-up: decode layers
  // 0.9-2.9 % and the K = 576 linear 3 % faster, T = 64 and K = 288 within
  // 1 % slower, the prefill chunk unchanged.)
  if (threadIdx.x == 0) ptx::griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Pair form: CTAs 2i and 2i+1 share every unit; the even one issues the MMAs.
  const uint32_t rank = PAIR ? ptx::cluster_rank() : 0u;
  const int arow = PAIR ? 128 * (int)rank : 0;  // this CTA's first token row in the unit
  const int u_first = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  // Pair form: every copy of both CTAs completes on the even CTA's barrier.
  const uint32_t lead_full = PAIR ? ptx::map_shared_rank(ptx::smem_u32(full), 0) : 0u;
  const int u_step = p.persistent ? (PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x) : p.units;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      // Unfused: the weight producer's arrival (with the weight bytes) and
      // the activation producer's arrival after its scale atom.  Fused: one
      // arrival per quantising warp; the copies are tracked by `landed`.
      // Pair form: the even CTA's barrier also takes the odd CTA's scale-atom
      // arrival and counts the bytes of both CTAs' copies; quantising pair
      // form: the atoms are copied too, so only the even CTA's two producers
      // arrive.
      ptx::mbar_init(&full[s], FUSED ? kEpiWarps : (PAIR ? (QUANT ? 2 : 3) : 2));
      ptx::mbar_init(&empty[s], 1);
      ptx::mbar_init(&landed[s], 1);
    }
    ptx::mbar_init(acc_full, 1);
    ptx::mbar_init(acc_empty, kEpiWarps * (PAIR ? 2 : 1));
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sf_full[b], 32);
      ptx::mbar_init(&sf_empty[b], 1);
    }
    ptx::mbar_init(mma_done, 1);
    if (QUANT)
      for (int i = 0; i < kQSlots + 1; ++i) ptx::mbar_init(&qfull[i], 1);
    abort_shared = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_act);
    ptx::prefetch_tmap(&tm_w);
    if (PAIR) ptx::prefetch_tmap(&tm_wsf);
    if (QUANT) {
      ptx::prefetch_tmap(map_asf(qmaps));
      ptx::prefetch_tmap(map_xq(qmaps));
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) ptx::cluster_sync();  // the peer's barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if constexpr (FUSED) {
    // ----------------------------------------------- producer (fused form)
    // `landed[s]` collects every copy of stage s: the weight tile and scale
    // atom (issued early, before waiting for the preceding kernel) and the
    // BF16 activation tile; its single arrival comes after all are issued.
    int it = 0, issued = 0;
    bool stop = false;
    auto issue_weights = [&](const Unit& w, int s, int kg) {
      ptx::mbar_expect_tx(&landed[s], C::X_TILE + C::W_SF_BYTES);
      ptx::tma_load_3d(smem + C::OFF_X + s * C::X_TILE, &tm_w, &landed[s], kg * 128, w.x0, w.g);
      ptx::bulk_load(smem + C::OFF_SFX + s * C::SFX_BYTES,
                     p.w_sf + (((size_t)w.g * p.KG + kg) * p.NB + w.x0 / 128) * kSfAtomBytes,
                     C::W_SF_BYTES, &landed[s]);
    };
    if (u_first < p.units) {
      const Unit w = decode_unit<SWAP, BN>(p, u_first);
      issued = min(w.nk, NSTAGE);
      if (lane == 0)
        for (int kk = 0; kk < issued; ++kk) issue_weights(w, kk, w.kg_begin + kk);
    }
    ptx::griddep_wait();
    for (int u = u_first; u < p.units && !stop; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      for (int kk = 0; kk < w.nk; ++kk) {
        const int s = it % NSTAGE;
        const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
        const int kg = w.kg_begin + kk;
        if (it >= issued) {
          if (*abort_flag || !ptx::mbar_wait_hint(&empty[s], ph ^ 1u, kWaitLimitNs, kPipeHintNs)) {
            if (!*abort_flag) watchdog(abort_flag, kWdProducer);
            stop = true;
            break;
          }
          if (lane == 0) issue_weights(w, s, kg);
          ++issued;
        }
        if (lane == 0) {
          ptx::mbar_expect_tx(&landed[s], C::STG_BYTES);
          ptx::tma_load_3d(smem + C::OFF_STG + s * C::STG_BYTES, &tm_act, &landed[s], kg * 128, w.g,
                           w.y0);
          ptx::mbar_arrive(&landed[s]);
        }
        __syncwarp();
        ++it;
      }
    }
    if (lane == 0)
      for (int j = it; j < issued; ++j) ptx::mbar_arrive(&landed[j % NSTAGE]);
    __syncwarp();
    for (int j = max(0, issued - NSTAGE); j < issued; ++j) {
      if (!ptx::mbar_wait(&landed[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, kWaitLimitNs)) {
        watchdog(abort_flag, kWdDrain);
        break;
      }
    }
    } else {
    // ----------------------------------------------------- weight producer
    // Stage bookkeeping (counters continue across units): stages < `issued`
    // have their weight copies in flight.  A stage's full barrier takes the
    // weight arrival (with its byte count) and the activation producer's
    // arrival after its scale atom (the activation tile's bytes announced
    // when that copy is issued); in the pair form the even CTA's barrier also
    // takes the odd CTA's atom arrival and counts both CTAs' bytes.  Weights
    // and activations are issued by two warps: one thread issues a TMA copy
    // only every few hundred cycles, so a single issuing thread cannot keep
    // the tensor cores fed.
    int it = 0, issued = 0;
    bool stop = false;
    auto issue_weights = [&](const Unit& w, int s, int kg) {
      uint8_t* wt = smem + (SWAP ? C::OFF_X + s * C::X_TILE : C::OFF_Y + s * C::Y_TILE);
      uint8_t* wsf = smem + (SWAP ? C::OFF_SFX + s * C::SFX_BYTES : C::OFF_SFY + s * C::SFY_BYTES);
      const int wtile0 = SWAP ? w.x0 : w.y0;
      const size_t atom0 = ((size_t)w.g * p.KG + kg) * p.NB + wtile0 / 128;
      if constexpr (PAIR) {
        // This CTA loads its half of the weight rows (lane 0) and the scale
        // atoms of the whole tile (lane 1: each thread issues only about one
        // TMA copy every few hundred cycles); the even CTA announces the
        // bytes of both CTAs.
        const uint32_t bar = lead_full + 8u * (uint32_t)s;
        if (lane == 0) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(&full[s], 2 * (C::Y_TILE + C::W_SF_BYTES));
          ptx::tma_load_3d_pair(wt, &tm_w, bar, kg * 128, wtile0 + C::Y_ROWS * (int)rank, w.g);
        } else {
          ptx::tma_load_2d_pair(wsf, &tm_wsf, bar, 0, (int)(atom0 * (kSfAtomBytes / 256)));
        }
      } else {
        ptx::mbar_arrive_expect_tx(&full[s], (SWAP ? C::X_TILE : C::Y_TILE) + C::W_SF_BYTES);
        ptx::tma_load_3d(wt, &tm_w, &full[s], kg * 128, wtile0, w.g);
        ptx::bulk_load(wsf, p.w_sf + atom0 * kSfAtomBytes, C::W_SF_BYTES, &full[s]);
      }
    };
    // Weight tiles and scales do not depend on the preceding kernel: the
    // first unit's first stages are issued before any wait, so the weight
    // stream starts while that kernel is still finishing.
    if (u_first < p.units) {
      const Unit w = decode_unit<SWAP, BN>(p, u_first);
      issued = min(w.nk, NSTAGE);
      if (lane < (PAIR ? 2 : 1))
        for (int kk = 0; kk < issued; ++kk) issue_weights(w, kk, w.kg_begin + kk);
    }
    for (int u = u_first; u < p.units && !stop; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      for (int kk = 0; kk < w.nk; ++kk) {
        const int s = it % NSTAGE;
        const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
        if (it >= issued) {
          if (*abort_flag || !ptx::mbar_wait_hint(&empty[s], ph ^ 1u, kWaitLimitNs, kPipeHintNs)) {
            if (!*abort_flag) watchdog(abort_flag, kWdProducer);
            stop = true;
            break;
          }
          if (lane < (PAIR ? 2 : 1)) issue_weights(w, s, w.kg_begin + kk);
          ++issued;
        }
        ++it;
      }
    }
    // Meet the activation producer; after an abort, give every stage that
    // has copies in flight the arrival it still lacks, so that its phase
    // completes once the copies have landed, then drain.
    ptx::named_sync(1, 64);
    const int act_issued = *act_done;
    if (lane == 0 && !(QUANT && rank != 0)) {
      for (int j = min(issued, act_issued); j < max(issued, act_issued); ++j) {
        if (PAIR && rank != 0)
          ptx::mbar_arrive_remote(lead_full + 8u * (uint32_t)(j % NSTAGE));
        else
          ptx::mbar_arrive(&full[j % NSTAGE]);
      }
    }
    __syncwarp();
    // Drain: every issued copy must have landed before exit (pair form: the
    // even CTA's barriers count both CTAs' copies, and the odd CTA stays
    // until the final cluster barrier).
    const int last = max(issued, act_issued);
    for (int j = max(0, last - NSTAGE); j < last && !(PAIR && rank != 0); ++j) {
      if (!ptx::mbar_wait(&full[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1u, kWaitLimitNs)) {
        watchdog(abort_flag, kWdDrain);
        break;
      }
    }
    }
  } else if (warp == kActWarp && QUANT) {
    // ------------------------------- activation producer (quantising form)
    // Per stage: the job counter of (this CTA's 128 tokens, K group) must
    // show every slice quantised.  Lane i reads (acquire) the counter of the
    // i-th next stage of the unit (one round trip for up to 32 stages; an
    // acquire load, unlike a fence, does not wait for the copies this warp
    // has in flight); lane 0 TMA-loads the codes and lane 1 the scale atom,
    // both counted on the even CTA's stage barrier.
    int it = 0;
    bool stop = false;
    uint8_t* tslot = smem + C::OFF_TK;
    uint64_t* tbar = qfull + kQSlots;
    uint32_t tphase = 0;
    ptx::griddep_wait();
    for (int u = u_first; u < p.units && !stop; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      const int fbase = (w.g * p.MB + w.x0 / 128 + (int)rank) * p.KG + w.kg_begin;
      int ready_end = 0;
      for (int kk = 0; kk < w.nk; ++kk) {
        const int s = it % NSTAGE;
        const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
        // Every decision of this loop is taken warp-uniformly (the polls
        // below use warp shuffles).
        const bool ok_empty =
            !*abort_flag && ptx::mbar_wait_hint(&empty[s], ph ^ 1u, kWaitLimitNs, kPipeHintNs);
        if (!__all_sync(0xffffffffu, ok_empty)) {
          if (lane == 0 && !*abort_flag) watchdog(abort_flag, kWdProducer);
          stop = true;
          break;
        }
        if (kk >= ready_end) {
          const int win = min(32, w.nk - kk);
          uint64_t t0 = 0;
          int nready = 0;
          while (true) {
            const bool rdy = lane < win && ptx::ld_acquire_gpu(p.qflags + fbase + kk + lane) >=
                                               (uint32_t)kQSlices;
            const uint32_t mask = __ballot_sync(0xffffffffu, rdy);
            nready = mask == 0xffffffffu ? 32 : __ffs(~mask) - 1;  // ready stages in a row
            if (nready > 0) break;
            // 1: another role aborted, 2: this wait ran out, 3: take the job over
            int give_up = 0;
            if (lane == 0) {
              const uint64_t now = ptx::globaltimer();
              if (*abort_flag)
                give_up = 1;
              else if (t0 == 0)
                t0 = now;
              else if (now - t0 > kWaitLimitNs)
                give_up = 2;
              else if (now - t0 > kTakeoverNs)
                give_up = 3;
            }
            give_up = __shfl_sync(0xffffffffu, give_up, 0);
            if (give_up == 3) {
              // The first stage not ready (stage kk): quantise its job here.
              if (!take_over_job(p, map_xq(qmaps), tslot, tbar, tphase, w.g, w.kg_begin + kk,
                                 (w.x0 / 128 + (int)rank) * 128, fbase + kk, lane)) {
                if (lane == 0) watchdog(abort_flag, kWdProducer);
                stop = true;
                break;
              }
              if (lane == 0) atomicAdd(&g_takeovers, 1u);
              t0 = 0;
              continue;
            }
            if (give_up) {
              if (give_up == 2 && lane == 0) watchdog(abort_flag, kWdProducer);
              stop = true;
              break;
            }
            __nanosleep(kFlagPollNs);
          }
          if (stop) break;
          // Each lane acquired its own stage's counter; the issuing lanes
          // order their copies after the warp's loads.
          __syncwarp();
          if (lane < 2) ptx::fence_proxy_async_global();
          ready_end = kk + nready;
        }
        const uint32_t bar = lead_full + 8u * (uint32_t)s;
        if (lane == 0) {
          if (rank == 0) ptx::mbar_arrive_expect_tx(&full[s], 2 * (C::X_TILE + C::SFX_BYTES));
          ptx::tma_load_3d_pair(smem + C::OFF_X + s * C::X_TILE, &tm_act, bar, (w.kg_begin + kk) * 128,
                                w.g, w.x0 + arow);
        } else if (lane == 1) {
          ptx::tma_load_2d_pair(smem + C::OFF_SFX + s * C::SFX_BYTES, map_asf(qmaps), bar, 0,
                                2 * (fbase + kk));
        }
        __syncwarp();
        ++it;
      }
    }
    if (lane == 0) *act_done = it;
    ptx::named_sync(1, 64);
  } else if (warp == kActWarp) {
    // ------------------------------------------------- activation producer
    // (The fused form quantises in the epilogue warps; this warp idles.)
    if constexpr (!FUSED) {
    int it = 0, ci = 0;
    bool stop = false;
    ptx::griddep_wait();  // the activation codes come from the preceding kernel
    for (int u = u_first; u < p.units && !stop; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      for (int kk = 0; kk < w.nk; ++kk) {
        const int b = ci & 1;
        const int s = it % NSTAGE;
        const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
        const int kg = w.kg_begin + kk;
        if (*abort_flag || !ptx::mbar_wait_hint(&empty[s], ph ^ 1u, kWaitLimitNs, kPipeHintNs)) {
          if (!*abort_flag) watchdog(abort_flag, kWdProducer);
          stop = true;
          break;
        }
        if ((kk % C::SF_CHUNK) == 0 &&
            !ptx::mbar_wait_hint(&sf_full[b], (uint32_t)(ci >> 1) & 1u, kWaitLimitNs, kPipeHintNs)) {
          watchdog(abort_flag, kWdProducer);
          stop = true;
          break;
        }
        if (lane == 0) {
          uint8_t* at = smem + (SWAP ? C::OFF_Y + s * C::Y_TILE : C::OFF_X + s * C::X_TILE);
          if constexpr (PAIR) {
            if (rank == 0) ptx::mbar_expect_tx(&full[s], 2 * C::X_TILE);
            ptx::tma_load_3d_pair(at, &tm_act, lead_full + 8u * (uint32_t)s, kg * 128, w.g,
                                  w.x0 + arow);
          } else {
            ptx::mbar_expect_tx(&full[s], SWAP ? C::Y_TILE : C::X_TILE);
            ptx::tma_load_3d(at, &tm_act, &full[s], kg * 128, w.g, SWAP ? w.y0 : w.x0);
          }
        }
        // Activation-scale atom: lane i writes the 16-byte line of rows
        // i, i+32, i+64, i+96 (one word each, the byte replicated four times).
        const uint8_t* col = csf + b * C::CSF_BYTES + (kk % C::SF_CHUNK) * 128;
        uint4 line;
        line.x = (uint32_t)col[lane] * 0x01010101u;
        line.y = (uint32_t)col[lane + 32] * 0x01010101u;
        line.z = (uint32_t)col[lane + 64] * 0x01010101u;
        line.w = (uint32_t)col[lane + 96] * 0x01010101u;
        uint8_t* asf = smem + (SWAP ? C::OFF_SFY + s * C::SFY_BYTES : C::OFF_SFX + s * C::SFX_BYTES);
        *reinterpret_cast<uint4*>(asf + lane * 16) = line;
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && rank != 0)
            ptx::mbar_arrive_remote(lead_full + 8u * (uint32_t)s);
          else
            ptx::mbar_arrive(&full[s]);
        }
        ++it;
        if ((kk % C::SF_CHUNK) == C::SF_CHUNK - 1 || kk == w.nk - 1) {
          if (lane == 0) ptx::mbar_arrive(&sf_empty[b]);
          ++ci;
        }
      }
    }
    if (lane == 0) *act_done = it;
    ptx::named_sync(1, 64);
    }
  } else if (warp == 1 && PAIR && rank != 0) {
    // Pair form, odd CTA: the even CTA issues every MMA and scale copy.
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    int it = 0, ti = 0;
    bool stop = false;
    for (int u = u_first; u < p.units && !stop; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      if constexpr (!PAIR) {
        if (*abort_flag ||
            !ptx::mbar_wait_hint(acc_empty, (uint32_t)(ti & 1) ^ 1u, kWaitLimitNs, kPipeHintNs)) {
          if (!*abort_flag) watchdog(abort_flag, kWdMma);
          break;
        }
        ptx::tc_fence_after();
      }
      for (int kk = 0; kk < w.nk; ++kk) {
        const int s = it % NSTAGE;
        const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
        if constexpr (PAIR) {
          // The gate warp has seen this stage land (and, before a unit's
          // first stage, the accumulator drained); meet it.
          ptx::named_sync(2, 64);
          if (!gate_go[it & 1]) {
            stop = true;
            break;
          }
        } else if (*abort_flag || !ptx::mbar_wait_hint(&full[s], ph, kWaitLimitNs, kPipeHintNs)) {
          if (!*abort_flag) watchdog(abort_flag, kWdMma);
          stop = true;
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
          const uint64_t adesc = ptx::smem_desc(xs, 16, 1024, ptx::kSwizzle128B);
          const uint64_t bdesc = ptx::smem_desc(ys, 16, 1024, ptx::kSwizzle128B);
          if constexpr (PAIR) {
            ptx::tmem_cp_32x128b_x4_pair(sfx_col, ptx::smem_desc(sfx, 128, 128, ptx::kSwizzleNone));
#pragma unroll
            for (int a = 0; a < C::Y_ATOMS; ++a)
              ptx::tmem_cp_32x128b_x4_pair(
                  sfy_col + 4 * a,
                  ptx::smem_desc(sfy + a * kSfAtomBytes, 128, 128, ptx::kSwizzleNone));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              ptx::mma_mxf8_pair(tmem, adesc + 2 * k, bdesc + 2 * k, C::IDESC, sfx_col, sfy_col,
                                 (kk > 0 || k > 0) ? 1u : 0u);
            ptx::tc_commit_pair_mc(&empty[s], 3);  // frees the stage in both CTAs
          } else {
            ptx::tmem_cp_32x128b_x4(sfx_col, ptx::smem_desc(sfx, 128, 128, ptx::kSwizzleNone));
#pragma unroll
            for (int a = 0; a < C::Y_ATOMS; ++a)
              ptx::tmem_cp_32x128b_x4(
                  sfy_col + 4 * a,
                  ptx::smem_desc(sfy + a * kSfAtomBytes, 128, 128, ptx::kSwizzleNone));
#pragma unroll
            for (int k = 0; k < 4; ++k)  // 4 x (K = 32 bytes) inside the 128-byte swizzle row
              ptx::mma_mxf8(tmem, adesc + 2 * k, bdesc + 2 * k, C::IDESC, sfx_col, sfy_col,
                            (kk > 0 || k > 0) ? 1u : 0u);
            ptx::tc_commit(&empty[s]);
          }
        }
        __syncwarp();
        ++it;
      }
      if (stop) break;
      if (lane == 0) {
        if constexpr (PAIR)
          ptx::tc_commit_pair_mc(acc_full, 3);
        else
          ptx::tc_commit(acc_full);
      }
      __syncwarp();
      ++ti;
    }
    // Every MMA and scale copy this warp issued must finish before TMEM is freed.
    if (lane == 0) {
      if constexpr (PAIR)
        ptx::tc_commit_pair_mc(mma_done, 1);
      else
        ptx::tc_commit(mma_done);
    }
    __syncwarp();
    if (!ptx::mbar_wait(mma_done, 0, kWaitLimitNs)) watchdog(abort_flag, kWdDrain);
  } else if (warp == 2 && !QUANT) {
    // ------------------------------------------------- activation scales
    // (The fused and quantising forms need no loader.)
    if constexpr (!FUSED && !QUANT) {
    int ci = 0;
    bool stop = false;
    for (int u = u_first; u < p.units && !stop; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      const int row0 = SWAP ? w.y0 : w.x0 + arow;
      if (u == u_first) ptx::griddep_wait();  // the scales come from the preceding kernel
      for (int c0 = 0; c0 < w.nk; c0 += C::SF_CHUNK) {
        const int b = ci & 1;
        if (*abort_flag ||
            !ptx::mbar_wait_hint(&sf_empty[b], ((uint32_t)(ci >> 1) & 1u) ^ 1u, kWaitLimitNs,
                                 kPipeHintNs)) {
          if (!*abort_flag) watchdog(abort_flag, kWdLoader);
          stop = true;
          break;
        }
        const int ng = min(C::SF_CHUNK, w.nk - c0);
        const int kg0 = w.kg_begin + c0;
        uint8_t* dst = csf + b * C::CSF_BYTES;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 32 * j + lane;
          const int t = row0 + r;
          const bool valid = r < C::ACT_ROWS && t < p.T;
          const uint8_t* src = p.a_sf + ((size_t)(valid ? t : 0) * p.G + w.g) * p.KG + kg0;
          if (valid && ((p.KG | kg0 | ng) & 15) == 0) {
            // 16-byte vectors: the row start and the chunk are 16-byte aligned.
            uint4 v[C::SF_CHUNK / 16];
#pragma unroll
            for (int q = 0; q < C::SF_CHUNK / 16; ++q)
              if (q * 16 < ng) v[q] = __ldg(reinterpret_cast<const uint4*>(src) + q);
#pragma unroll
            for (int q = 0; q < C::SF_CHUNK / 16; ++q) {
              if (q * 16 >= ng) break;
              const uint32_t wv[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
              for (int e = 0; e < 16; ++e)
                dst[(q * 16 + e) * 128 + r] = (uint8_t)(wv[e >> 2] >> (8 * (e & 3)));
            }
          } else if (valid) {
            for (int q = 0; q < ng; ++q) dst[q * 128 + r] = __ldg(src + q);
          } else {
            for (int q = 0; q < ng; ++q) dst[q * 128 + r] = 127;
          }
        }
        ptx::mbar_arrive(&sf_full[b]);  // every lane: its own stores are released
        ++ci;
      }
    }
    }
  } else if (warp == (QUANT ? kQGateWarp : kGateWarp)) {
    // ---------------------------------------------------- gate (pair form)
    // Waits, for the even CTA's MMA warp, on the accumulator at each unit's
    // start and on each stage's full barrier, then meets the MMA warp at a
    // named barrier.  Both warps pass that barrier exactly once per stage
    // (or once more with "stop" after a failed bounded wait, then both
    // leave), and the go flag alternates between two slots so that it is
    // never rewritten before the MMA warp has read it.
    if constexpr (PAIR) {
      if (rank == 0) {
        int it = 0, ti = 0;
        bool ok = true;
        for (int u = u_first; u < p.units && ok; u += u_step) {
          const Unit w = decode_unit<SWAP, BN>(p, u);
          ok = !*abort_flag &&
               ptx::mbar_wait_hint(acc_empty, (uint32_t)(ti & 1) ^ 1u, kWaitLimitNs, kPipeHintNs);
          for (int kk = 0; kk < w.nk; ++kk) {
            const int s = it % NSTAGE;
            const uint32_t ph = (uint32_t)(it / NSTAGE) & 1u;
            ok = ok && !*abort_flag && ptx::mbar_wait_hint(&full[s], ph, kWaitLimitNs, kPipeHintNs);
            if (lane == 0) gate_go[it & 1] = ok ? 1 : 0;
            ptx::named_sync(2, 64);
            if (!ok) break;
            ++it;
          }
          ++ti;
        }
        if (!ok && !*abort_flag) watchdog(abort_flag, kWdMma);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quadrant this warp may access
    const int h = (warp - kEpiWarp0) >> 2;        // which half of the columns
    const int r = q * 32 + lane;                  // accumulator row (TMEM lane)
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + h * C::HALF;
    float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // split-K receive buffer
    int ti = 0;
    int itq = 0;  // stage counter of the fused activation quantisation
    if constexpr (FUSED) {
      // Scale-atom rows past the token tile (BN < 128) never change: 127.
      const int te = threadIdx.x - kEpiWarp0 * 32;
      for (int i = te; i < NSTAGE * (128 - BN); i += kEpiWarps * 32) {
        const int s = i / (128 - BN);
        const int rr = BN + i % (128 - BN);
        *reinterpret_cast<uint32_t*>(smem + C::OFF_SFY + s * C::SFY_BYTES + (rr & 31) * 16 +
                                     ((rr >> 5) & 3) * 4) = 0x7F7F7F7Fu;
      }
      ptx::griddep_wait();  // positions (and x, via TMA) come from preceding kernels
    }
    if constexpr (QUANT) {
      // Quantising pair form: between accumulator drains (which go first)
      // this warp quantises its activation slices; every wait is a
      // non-blocking test, bounded in wall time while nothing is ready.
      // This warp quantises slice qw (rows t0 + 16 qw + [0, 16)) of every job
      // of its CTA, in job order, from its own slot: it copies the next
      // job's slice into the slot with TMA as soon as the current one is
      // read, and prefetches the slice kQPrefetch jobs ahead into L2.
      // Publication: every kQPublish slices (each of the first few, when
      // nothing else is ready, and the last) the warp makes its earlier
      // slices' writes visible at gpu scope and raises their jobs' counters,
      // just before the current slice's stores, so that the fence finds the
      // earlier stores done.
      const int qw = warp - kEpiWarp0;
      // Drains this warp's quarter of the unit's accumulator (after its
      // acc_full phase) and stores it, as the plain pair form's loop below
      // does.  (The two copies are kept apart: a drain shared by every form's
      // epilogue measured 0.8 us per layer slower in the few-token forms,
      // which never drain this way.)
      auto pair_drain = [&](const Unit& w) {
        // Drain 32 columns at a time and keep them as packed BF16 pairs (RNE,
        // as in the other forms), so that the CTA fits its register budget;
        // the accumulator is released as soon as it is read.
        uint32_t pk[C::HALF / 2];
  #pragma unroll
        for (int c = 0; c < C::HALF / 32; ++c) {
          uint32_t t32[32];
          ptx::tmem_ld_32x32b_x32(trow + c * 32, t32);
          ptx::tmem_ld_wait();
  #pragma unroll
          for (int j = 0; j < 16; ++j) pk[c * 16 + j] = pack_bf16x2(t32[2 * j], t32[2 * j + 1]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)  // the accumulator may be overwritten now
          ptx::mbar_arrive_remote(ptx::map_shared_rank(ptx::smem_u32(acc_empty), 0));
        // Rows of a lane are 16 KB apart in the output, so each warp stages
        // 32 rows x 32 columns in shared memory and one lane stores the box
        // with TMA (full lines, no per-lane scattered stores; rows past T
        // and columns past N are clipped by the copy).
        const int c0 = h * C::HALF;
        uint8_t* buf = smem + C::OFF_OUT + (warp - kEpiWarp0) * C::OUT_TILE;
  #pragma unroll
        for (int c = 0; c < C::HALF / 32; ++c) {
          if (lane == 0) ptx::bulk_wait_read<0>();  // the previous chunk's store has read it
          __syncwarp();
  #pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 64 + j * 16) =
                make_uint4(pk[c * 16 + j * 4 + 0], pk[c * 16 + j * 4 + 1], pk[c * 16 + j * 4 + 2],
                           pk[c * 16 + j * 4 + 3]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tm_out, buf, w.y0 + c0 + c * 32, w.g, w.x0 + arow + q * 32);
            ptx::bulk_commit_group();
          }
        }
      };
      uint8_t* qslot = smem + C::OFF_QX + qw * kQSliceBytes;
      // x is read once: its lines leave L2 first, ahead of the codes, which
      // the CTA pairs read back shortly after.
      const uint64_t x_policy = ptx::policy_evict_first();
      // The y_tiles units of a token block share its jobs and are
      // consecutive, so their ordinals (in their pairs) differ by at most
      // ceil((y_tiles - 1) / u_step).  With a lead of at least that, the
      // jobs that the pair furthest behind is multiplying are always
      // allowed, wherever they fall: the pairs cannot wait on each other in
      // a cycle.
      const int q_lead = max(kQLead, (p.y_tiles - 1 + u_step - 1) / u_step);
      uint64_t* qbar = &qfull[qw];
      QJob j;
      bool have = u_first < p.q_lazy_from && qjob_first(p, u_first, u_step, (int)rank, j);
      int k = 0, npend = 0;  // slices copied into the slot; counters not yet raised
      int pend[kQPublish];
      auto pos_of = [&](const QJob& jj) -> int64_t {
        const int t = jj.t0 + kQRows * qw + (lane & 15);
        return (p.R > 0 && t < p.T) ? __ldg(p.pos + t) : 0;
      };
      auto load_slice = [&](const QJob& jj) {
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(qbar, kQSliceBytes);
          ptx::tma_load_3d_hint(qslot, map_xq(qmaps), qbar, jj.kg * 128, jj.g, jj.t0 + kQRows * qw,
                                x_policy);
        }
      };
      QJob jp = j;  // L2 prefetch cursor
      bool pmore = have;
      auto prefetch_next = [&]() {
        if (pmore) pmore = qjob_next(p, u_step, (int)rank, jp);
        if (pmore && lane == 0) ptx::tma_prefetch_3d(map_xq(qmaps), jp.kg * 128, jp.g, jp.t0 + kQRows * qw);
      };
      auto q_publish = [&]() {
        // The codes and atom words are read by other CTAs through TMA.
        ptx::fence_proxy_async_global();
        ptx::fence_acq_rel_gpu();
        __syncwarp();
        if (lane < npend) {
          int f = pend[0];
#pragma unroll
          for (int i = 1; i < kQPublish; ++i)
            if (lane == i) f = pend[i];
          ptx::red_add_relaxed_gpu(p.qflags + f, 1u);
        }
        npend = 0;
      };
      ptx::griddep_wait();  // x, the positions and the cleared counters come from preceding work
      int64_t pl = 0;
      if (have) {
        pl = pos_of(j);
        load_slice(j);
        for (int i = 0; i < kQPrefetch; ++i) prefetch_next();
      }
      auto q_ready = [&]() {
        return __all_sync(0xffffffffu, ptx::mbar_test(qbar, (uint32_t)k & 1u));
      };
      auto q_step = [&]() {
        const QJob jc = j;
        const int64_t plc = pl;
        const uint32_t badmask =
            __ballot_sync(0xffffffffu, p.R > 0 && jc.t0 + kQRows * qw + (lane & 15) < p.T &&
                                           (plc < 0 || plc >= p.max_pos)) & 0xFFFFu;
        QJob jn = j;
        const bool more = qjob_next(p, u_step, (int)rank, jn);
        const int64_t pn = more ? pos_of(jn) : 0;
        const bool due = npend == kQPublish || (npend > 0 && k < kQPublish);
        // Once this warp's reads of the slot are done: copy the next slice in.
        auto refill = [&]() {
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (more) load_slice(jn);
          prefetch_next();
        };
        if (p.R > 0 && jc.kg == p.KG - 1) {
          if (due) q_publish();
          qslice_rope(p, jc, qw, qslot, lane, badmask, plc);
          refill();
        } else {
          qslice_plain(p, jc, qw, qslot, lane, badmask, refill, [&]() {
            if (due) q_publish();
          });
        }
        if (badmask != 0 && jc.kg == 0 && lane == 0 && p.err_flag != nullptr)
          atomicOr(p.err_flag, MXQ_DEVERR_POSITION);
#pragma unroll
        for (int i = 0; i < kQPublish; ++i)
          if (i == npend) pend[i] = jc.f;
        ++npend;
        ++k;
        j = jn;
        pl = pn;
        have = more;
      };
      int u = u_first;
      uint64_t idle0 = 0;
      bool aborted = false;
      while (u < p.units || have) {
        if (u < p.units &&
            __all_sync(0xffffffffu, ptx::mbar_test(acc_full, (uint32_t)(ti & 1)))) {
          ptx::tc_fence_after();
          pair_drain(decode_unit<SWAP, BN>(p, u));
          ++ti;
          u += u_step;
          idle0 = 0;
          continue;
        }
        // A job of the unit of ordinal n (this pair's n-th unit) is
        // quantised once this warp has drained n - q_lead units: the codes
        // then wait in L2 for a short time only, instead of being written
        // back and read again from DRAM.
        if (have && (j.u - u_first) / u_step <= ti + q_lead && q_ready()) {
          q_step();
          idle0 = 0;
          continue;
        }
        if (npend > 0) {  // nothing ready: publish what is pending now
          q_publish();
          continue;
        }
        int give_up = 0;  // 1: another role aborted, 2: nothing became ready in time
        if (lane == 0) {
          const uint64_t now = ptx::globaltimer();
          if (*abort_flag)
            give_up = 1;
          else if (idle0 == 0)
            idle0 = now;
          else if (now - idle0 > kWaitLimitNs)
            give_up = 2;
        }
        give_up = __shfl_sync(0xffffffffu, give_up, 0);
        if (give_up) {
          if (give_up == 2 && lane == 0) watchdog(abort_flag, kWdEpilogue);
          aborted = true;
          break;
        }
        __nanosleep(kEpiPollNs);
      }
      if (!aborted && npend > 0) q_publish();
      // A copy still in flight into the slot (after an abort) lands before
      // the CTA may retire.
      if (have && !ptx::mbar_wait(qbar, (uint32_t)k & 1u, kWaitLimitNs) && lane == 0)
        watchdog(abort_flag, kWdDrain);
    } else
    for (int u = u_first; u < p.units; u += u_step) {
      const Unit w = decode_unit<SWAP, BN>(p, u);
      if constexpr (FUSED) {
        // ---------------------------------------- fused activation quantisation
        // Half-warp per token: token slot = 16*pass + 2*e + half, lane `sub`
        // holds elements [8*sub, 8*sub+8) of the stage's 128-wide group.
        constexpr int PASSES = BN / 16;
        const int e = warp - kEpiWarp0;
        const int sub = lane & 15;
        const int hw = lane >> 4;
        const bool has_rope = p.R > 0 && w.kg_begin + w.nk == p.KG;
        const int first = 16 - (p.R >> 3);
        const int dist = p.R >> 4;
        const bool rope_lane = p.R > 0 && sub >= first;
        const bool lower = sub < first + dist;
        const int partner = rope_lane ? (lower ? sub + dist : sub - dist) : sub;
        bool bad[PASSES];
        uint4 cw[PASSES], sw[PASSES];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
          const int t = w.y0 + 16 * ps + 2 * e + hw;
          int64_t pp = 0;
          bad[ps] = false;
          cw[ps] = make_uint4(0, 0, 0, 0);
          sw[ps] = make_uint4(0, 0, 0, 0);
          if (p.R > 0 && t < p.T) {
            pp = __ldg(p.pos + t);
            bad[ps] = pp < 0 || pp >= p.max_pos;
            if (has_rope && rope_lane && !bad[ps]) {
              const int i0 = (sub - first - (lower ? 0 : dist)) * 8;
              cw[ps] = __ldg(reinterpret_cast<const uint4*>(p.cos_tab + pp * p.cs_ld + i0));
              sw[ps] = __ldg(reinterpret_cast<const uint4*>(p.sin_tab + pp * p.cs_ld + i0));
            }
            if (bad[ps] && sub == 0 && w.x0 == 0 && w.split == 0 && p.err_flag != nullptr)
              atomicOr(p.err_flag, MXQ_DEVERR_POSITION);
          }
        }
        bool qstop = false;
        for (int kk = 0; kk < w.nk; ++kk) {
          const int s = itq % NSTAGE;
          const uint32_t ph = (uint32_t)(itq / NSTAGE) & 1u;
          const bool ok_wait =
              !*abort_flag && ptx::mbar_wait_hint(&landed[s], ph, kWaitLimitNs, kPipeHintNs);
          if (!__all_sync(0xffffffffu, ok_wait)) {
            if (!*abort_flag) watchdog(abort_flag, kWdEpilogue);
            qstop = true;
            break;
          }
          const bool rope = has_rope && w.kg_begin + kk == p.KG - 1;
          const uint8_t* stg = smem + C::OFF_STG + s * C::STG_BYTES;
          uint8_t* codes = smem + C::OFF_Y + s * C::Y_TILE;
          uint8_t* atom = smem + C::OFF_SFY + s * C::SFY_BYTES;
#pragma unroll
          for (int ps = 0; ps < PASSES; ++ps) {
            const int slot = 16 * ps + 2 * e + hw;
            const bool valid = w.y0 + slot < p.T;
            const uint4 v = *reinterpret_cast<const uint4*>(stg + slot * 256 + sub * 16);
            float y[8];
            unpack8(v, y);
            if (rope) {
              const int src = (hw << 4) | partner;
              uint4 pv;
              pv.x = __shfl_sync(0xffffffffu, v.x, src);
              pv.y = __shfl_sync(0xffffffffu, v.y, src);
              pv.z = __shfl_sync(0xffffffffu, v.z, src);
              pv.w = __shfl_sync(0xffffffffu, v.w, src);
              if (rope_lane && valid && !bad[ps]) {
                float xp[8];
                unpack8(pv, xp);
                inv_rope8(y, xp, cw[ps], sw[ps], lower);
              }
            }
            const float amax = half_warp_amax(y);
            uint32_t sbyte;
            uint2 q8 = encode8(y, amax, &sbyte);
            if (!valid) {  // padding token of the tile
              q8 = make_uint2(0, 0);
              sbyte = 127;
            }
            if (bad[ps]) {  // a token with an invalid position is zeroed
              q8 = make_uint2(0, 0);
              sbyte = 0;
            }
            // 128-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8).
            const int c16 = sub >> 1;
            *reinterpret_cast<uint2*>(codes + slot * 128 + ((c16 ^ (slot & 7)) << 4) + ((sub & 1) << 3)) =
                q8;
            if (sub == 0)
              *reinterpret_cast<uint32_t*>(atom + (slot >> 7) * kSfAtomBytes + (slot & 31) * 16 +
                                           ((slot >> 5) & 3) * 4) = sbyte * 0x01010101u;
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&full[s]);
          ++itq;
        }
        if (qstop) break;
      }
      const bool waited =
          !*abort_flag && ptx::mbar_wait_hint(acc_full, (uint32_t)(ti & 1), kWaitLimitNs, kPipeHintNs);
      if (!__all_sync(0xffffffffu, waited)) {
        if (!*abort_flag) watchdog(abort_flag, kWdEpilogue);
        break;
      }
      ptx::tc_fence_after();
      if constexpr (PAIR) {
        // Drain 32 columns at a time and keep them as packed BF16 pairs (RNE,
        // as in the other forms), so that the 13-warp CTA fits its register
        // budget; the accumulator is released as soon as it is read.
        uint32_t pk[C::HALF / 2];
  #pragma unroll
        for (int c = 0; c < C::HALF / 32; ++c) {
          uint32_t t32[32];
          ptx::tmem_ld_32x32b_x32(trow + c * 32, t32);
          ptx::tmem_ld_wait();
  #pragma unroll
          for (int j = 0; j < 16; ++j) pk[c * 16 + j] = pack_bf16x2(t32[2 * j], t32[2 * j + 1]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0)  // the accumulator may be overwritten now
          ptx::mbar_arrive_remote(ptx::map_shared_rank(ptx::smem_u32(acc_empty), 0));
        // Rows of a lane are 16 KB apart in the output, so each warp stages
        // 32 rows x 32 columns in shared memory and one lane stores the box
        // with TMA (full lines, no per-lane scattered stores; rows past T
        // and columns past N are clipped by the copy).
        const int c0 = h * C::HALF;
        uint8_t* buf = smem + C::OFF_OUT + (warp - kEpiWarp0) * C::OUT_TILE;
  #pragma unroll
        for (int c = 0; c < C::HALF / 32; ++c) {
          if (lane == 0) ptx::bulk_wait_read<0>();  // the previous chunk's store has read it
          __syncwarp();
  #pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 64 + j * 16) =
                make_uint4(pk[c * 16 + j * 4 + 0], pk[c * 16 + j * 4 + 1], pk[c * 16 + j * 4 + 2],
                           pk[c * 16 + j * 4 + 3]);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tm_out, buf, w.y0 + c0 + c * 32, w.g, w.x0 + arow + q * 32);
            ptx::bulk_commit_group();
          }
        }
        ++ti;
        continue;
      }
      uint32_t v[C::HALF];
      if constexpr (C::HALF % 32 == 0) {
#pragma unroll
        for (int c = 0; c < C::HALF / 32; ++c) ptx::tmem_ld_32x32b_x32(trow + c * 32, v + c * 32);
      } else {
#pragma unroll
        for (int c = 0; c < C::HALF / 8; ++c) ptx::tmem_ld_32x32b_x8(trow + c * 8, v + c * 8);
      }
      ptx::tmem_ld_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(acc_empty);  // the accumulator may be overwritten now
      ++ti;
      if (w.nk == 0) {
#pragma unroll
        for (int j = 0; j < C::HALF; ++j) v[j] = 0u;  // an empty K slice contributes zero
      }
      const int c0 = h * C::HALF;
      if (!SWAP) {
        const int t = w.x0 + arow + r;
        if (t < p.T) {
          __nv_bfloat16* orow = p.out + ((size_t)t * p.G + w.g) * p.N + w.y0 + c0;
#pragma unroll
          for (int c = 0; c < C::HALF / 8; ++c) {
            if (w.y0 + c0 + c * 8 < p.N) {
              uint4 o;
              o.x = pack_bf16x2(v[c * 8 + 0], v[c * 8 + 1]);
              o.y = pack_bf16x2(v[c * 8 + 2], v[c * 8 + 3]);
              o.z = pack_bf16x2(v[c * 8 + 4], v[c * 8 + 5]);
              o.w = pack_bf16x2(v[c * 8 + 6], v[c * 8 + 7]);
              *reinterpret_cast<uint4*>(orow + c * 8) = o;
            }
          }
        }
      } else if (p.splits == 1) {
        const int n = w.x0 + r;
#pragma unroll
        for (int j = 0; j < C::HALF; ++j) {
          const int t = w.y0 + c0 + j;
          if (t < p.T && n < p.N)
            p.out[((size_t)t * p.G + w.g) * p.N + n] = __float2bfloat16_rn(__uint_as_float(v[j]));
        }
      } else {
        // Split K: push this row's fp32 partial straight into the receive
        // buffer of the cluster CTA that owns the row (slot = our rank).
        const int rps = (C::BM + p.splits - 1) / p.splits;
        const int owner = r / rps;
        const uint32_t dst = ptx::map_shared_rank(
            ptx::smem_u32(red + ((w.split * rps + (r - owner * rps)) * C::PART_PITCH + c0)),
            (uint32_t)owner);
#pragma unroll
        for (int j = 0; j < C::HALF; j += 4)
          ptx::st_shared_cluster_f32x4(dst + j * 4, __uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                       __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      }
    }
  }

  if constexpr (PAIR) {
    // The output stores must be complete (and their shared-memory sources
    // read) before the CTA retires.
    if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps && lane == 0) ptx::bulk_wait_all();
  }
  __syncthreads();
  if (SWAP && p.splits > 1) {
    // Deterministic split-K reduction over the cluster (one unit per CTA).
    // Every CTA pushed its partial rows to their owners before the barrier;
    // after it, CTA `split` sums the rows it owns over ranks 0..splits-1 in
    // order, from its own shared memory, and nobody touches a peer again.
    const Unit w = decode_unit<SWAP, BN>(p, u_first);
    ptx::cluster_sync();
    const int rps = (C::BM + p.splits - 1) / p.splits;
    const int r_begin = w.split * rps;
    const int nrows = min(C::BM, r_begin + rps) - r_begin;
    const int tv = min(BN, p.T - w.y0);
    if (!*abort_flag && nrows > 0 && tv > 0) {
      // Work item = (row, 4 consecutive tokens), rows fastest so that the
      // BF16 stores of a warp are contiguous along n.
      const float* red = reinterpret_cast<const float*>(smem + C::OFF_RED);
      const int tv4 = (tv + 3) >> 2;
      for (int e = threadIdx.x; e < nrows * tv4; e += C::THREADS) {
        const int tl = (e / nrows) * 4;
        const int rr = e % nrows;
        float4 acc = *reinterpret_cast<const float4*>(red + rr * C::PART_PITCH + tl);
        for (int rk = 1; rk < p.splits; ++rk) {
          const float4 pv =
              *reinterpret_cast<const float4*>(red + (rk * rps + rr) * C::PART_PITCH + tl);
          acc.x += pv.x;
          acc.y += pv.y;
          acc.z += pv.z;
          acc.w += pv.w;
        }
        const int n = w.x0 + r_begin + rr;
        if (n < p.N) {
          const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
          __nv_bfloat16* o = p.out + ((size_t)(w.y0 + tl) * p.G + w.g) * p.N + n;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (tl + j < tv) o[(size_t)j * p.G * p.N] = __float2bfloat16_rn(a4[j]);
        }
      }
    }
  }
  if constexpr (PAIR) ptx::cluster_sync();  // no CTA leaves while its peer may still use it
  if (warp == 1) {
    ptx::tc_fence_after();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// A kernel that waits on an mbarrier nobody arrives at: the bounded wait must
// give up after `limit_ns` and record the expiry in the watchdog word.
__global__ void watchdog_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, limit_ns)) atomicOr(&g_watchdog, 1u << 31);
  __syncthreads();
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

// 3-D tensor map with zero fill outside the tensor: uint8 codes with
// 128-byte rows swizzled (MMA operands), or BF16 rows unswizzled (the fused
// form's activation staging).
bool encode_3d(CUtensorMap* m, const void* base, bool bf16, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   bf16 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D uint8 map over scale atoms (the prepared weight scales, or the
// activation atoms of the quantising form), 256-byte rows (two per 512-byte
// atom), boxes of `rows` rows: the pair form's scale-atom copies.
bool encode_scale_rows(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {256, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool SWAP, bool FUSED, int BN, int NSTAGE, bool PAIR = false, bool QUANT = false>
cudaError_t launch_cfg(const void* a, const uint8_t* w, BmmArgs args, int num_sms,
                       cudaStream_t s, const char** why) {
  using C = Cfg<SWAP, FUSED, BN, NSTAGE, PAIR, QUANT>;
  const uint64_t K = args.K, G = args.G, T = args.T, N = args.N;
  CUtensorMap tm_act, tm_w;
  const uint32_t act_box = SWAP ? BN : C::BM;
  const uint32_t w_box = SWAP ? C::BM : C::Y_ROWS;
  const uint64_t esz = FUSED ? 2 : 1;  // fused form: x is BF16
  CUtensorMap tm_wsf = {}, tm_out = {}, tm_asf = {}, tm_xq = {};
  const uint64_t atoms = G * (uint64_t)args.KG * (uint64_t)args.NB;
  if (!encode_3d(&tm_act, a, FUSED, K, G, T, K * esz, G * K * esz, 128, 1, act_box) ||
      !encode_3d(&tm_w, w, false, K, N, G, K, N * K, 128, w_box, 1) ||
      (PAIR && !encode_scale_rows(&tm_wsf, args.w_sf, atoms * (kSfAtomBytes / 256),
                                  (uint32_t)(C::W_SF_BYTES / 256))) ||
      // Output [T][G][N] BF16, 32 x 32 boxes of one group (pair-form epilogue).
      (PAIR && !encode_3d(&tm_out, args.out, true, N, G, T, N * 2, G * N * 2, 32, 1, 32)) ||
      // Activation scale atoms written by the quantising warps, as 256-byte
      // rows (two per atom).
      (QUANT && !encode_scale_rows(&tm_asf, args.qatoms,
                                   G * (uint64_t)args.MB * (uint64_t)args.KG * (kSfAtomBytes / 256),
                                   (uint32_t)(kSfAtomBytes / 256))) ||
      // The BF16 activation [T][G][K], 32-row x 128-value slices.
      (QUANT && !encode_3d(&tm_xq, args.xq, true, K, G, T, K * 2, G * K * 2, 128, 1, kQRows))) {
    *why = "cuTensorMapEncodeTiled failed (driver entry point missing or arguments rejected)";
    return cudaErrorInvalidValue;
  }
  auto kern = bmm_a8w8_kernel<SWAP, FUSED, BN, NSTAGE, PAIR, QUANT>;
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
  if (SWAP) {
    // Split K so that about one wave of CTAs streams the weights (deterministic
    // rank-order reduction over a cluster of at most 8).
    const int base = args.x_tiles * args.y_tiles * args.G;
    int splits = (num_sms * C::CTAS_PER_SM) / (base > 0 ? base : 1);
    splits = splits < 1 ? 1 : (splits > 8 ? 8 : splits);
    splits = splits > args.KG ? args.KG : splits;
    // With at most three K groups per tile the cluster reduction costs more
    // than spreading them saves (measured: K = 288, 4.2 -> 3.6 us per call).
    if (args.KG <= 3) splits = 1;
    args.kg_per_split = (int)ceil_div(args.KG, splits);
    args.splits = (int)ceil_div(args.KG, args.kg_per_split);
    if (args.splits > 1 && args.splits * (int)ceil_div(C::BM, args.splits) > C::RED_ROWS) {
      *why = "split-K receive buffer too small for this split count";
      return cudaErrorInvalidValue;
    }
  }
  args.units = args.G * args.x_tiles * args.y_tiles * args.splits;
  args.persistent = args.splits == 1 ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  // Programmatic dependent launch: the grid may start while the preceding
  // kernel on the stream finishes; it waits (griddepcontrol.wait) before
  // reading anything that kernel produced.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int cluster = PAIR ? 2 : args.splits;
  if (cluster > 1) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = (unsigned)cluster;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    ++cfg.numAttrs;
  }

  int grid = args.units;
  if (PAIR) {
    // One persistent CTA pair per co-resident cluster slot (the SM pairs the
    // GPCs can form), each pair walking the units.
    static std::atomic<int> pair_slots[64];
    int slots = pair_slots[dev & 63].load(std::memory_order_acquire);
    if (slots == 0) {
      cfg.gridDim = dim3(2u * (unsigned)(num_sms / 2), 1, 1);
      e = cudaOccupancyMaxActiveClusters(&slots, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (slots <= 0) {
        *why = "no CTA pair fits on this device";
        return cudaErrorInvalidConfiguration;
      }
      pair_slots[dev & 63].store(slots, std::memory_order_release);
    }
    const int cap = g_pair_limit.load(std::memory_order_relaxed);
    if (cap > 0 && cap < slots) slots = cap;
    grid = 2 * (args.units < slots ? args.units : slots);
  } else if (args.persistent) {
    const int slots = num_sms * C::CTAS_PER_SM;
    grid = args.units < slots ? args.units : slots;
  }
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  QuantMapsT<QUANT> qmaps{};
  if constexpr (QUANT) {
    qmaps.asf = tm_asf;
    qmaps.xq = tm_xq;
  }
  return cudaLaunchKernelEx(&cfg, kern, tm_act, tm_w, tm_wsf, tm_out, qmaps, args);
}

}  // namespace

cudaError_t launch_bmm_a8w8(const uint8_t* a, const uint8_t* a_sf, const uint8_t* w,
                            const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                            int num_sms, cudaStream_t s, const char** why) {
  BmmArgs args = {};
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
    args.x_span = 128;
    args.x_tiles = (int)ceil_div(N, 128);
    args.y_tiles = 1;
    if (T <= 16) return launch_cfg<true, false, 16, 5>(a, w, args, num_sms, s, why);
    if (T <= 32) return launch_cfg<true, false, 32, 4>(a, w, args, num_sms, s, why);
    if (T <= 64) return launch_cfg<true, false, 64, 4>(a, w, args, num_sms, s, why);
    return launch_cfg<true, false, 128, 4>(a, w, args, num_sms, s, why);
  }
  // Many tokens: CTA pairs, 256 tokens x 256 weight rows per unit.
  args.x_span = 256;
  args.x_tiles = (int)ceil_div(T, 256);
  args.y_tiles = (int)ceil_div(N, 256);
  args.splits = 1;
  args.kg_per_split = args.KG;
  return launch_cfg<false, false, 256, 6, true>(a, w, args, num_sms, s, why);
}

cudaError_t launch_wo_a_fused(const void* x, const int64_t* pos, const void* cos, const void* sin,
                              int64_t cs_ld, int64_t max_pos, int R, const uint8_t* w,
                              const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                              int32_t* err_flag, int num_sms, cudaStream_t s, const char** why) {
  BmmArgs args = {};
  args.w_sf = w_sf;
  args.out = reinterpret_cast<__nv_bfloat16*>(out);
  args.T = (int)T;
  args.G = G;
  args.N = N;
  args.K = K;
  args.KG = (int)ceil_div(K, kGroup);
  args.NB = (int)sf_row_blocks(N);
  args.pos = pos;
  args.cos_tab = reinterpret_cast<const uint16_t*>(cos);
  args.sin_tab = reinterpret_cast<const uint16_t*>(sin);
  args.cs_ld = cs_ld;
  args.max_pos = max_pos;
  args.R = R;
  args.err_flag = err_flag;
  args.x_span = 128;
  args.x_tiles = (int)ceil_div(N, 128);
  args.y_tiles = 1;
  if (T <= 16) return launch_cfg<true, true, 16, 4>(x, w, args, num_sms, s, why);
  return launch_cfg<true, true, 32, 3>(x, w, args, num_sms, s, why);
}

cudaError_t launch_wo_a_prefill(const void* x, const int64_t* pos, const void* cos, const void* sin,
                                int64_t cs_ld, int64_t max_pos, int R, const uint8_t* w,
                                const uint8_t* w_sf, void* out, int64_t T, int G, int N, int K,
                                int32_t* err_flag, void* ws, int num_sms, cudaStream_t s,
                                const char** why) {
  BmmArgs args = {};
  args.w_sf = w_sf;
  args.out = reinterpret_cast<__nv_bfloat16*>(out);
  args.T = (int)T;
  args.G = G;
  args.N = N;
  args.K = K;
  args.KG = (int)ceil_div(K, kGroup);
  args.NB = (int)sf_row_blocks(N);
  args.pos = pos;
  args.cos_tab = reinterpret_cast<const uint16_t*>(cos);
  args.sin_tab = reinterpret_cast<const uint16_t*>(sin);
  args.cs_ld = cs_ld;
  args.max_pos = max_pos;
  args.R = R;
  args.err_flag = err_flag;
  args.x_span = 256;
  args.x_tiles = (int)ceil_div(T, 256);
  args.y_tiles = (int)ceil_div(N, 256);
  args.splits = 1;
  args.kg_per_split = args.KG;
  args.MB = 2 * args.x_tiles;
  args.q_lazy_from = g_lazy_from.load(std::memory_order_relaxed);
  const WoaPrefillLayout l = woa_prefill_layout(T, G, K);
  uint8_t* base = static_cast<uint8_t*>(ws);
  args.xq = reinterpret_cast<const uint16_t*>(x);
  args.qcodes = base + l.codes;
  args.qatoms = base + l.atoms;
  args.qflags = reinterpret_cast<uint32_t*>(base + l.flags);
  // The job counters start at zero on every call (a counter is raised once
  // per quantising warp and job, and read against that count).
  cudaError_t e = cudaMemsetAsync(args.qflags, 0, l.total - l.flags, s);
  if (e != cudaSuccess) return e;
  return launch_cfg<false, false, 256, 5, true, true>(args.qcodes, w, args, num_sms, s, why);
}

int set_pair_limit(int pairs) { return g_pair_limit.exchange(pairs < 0 ? 0 : pairs); }
int set_lazy_pairs(int from) { return g_lazy_from.exchange(from < 0 ? (1 << 30) : from); }

cudaError_t watchdog_read(uint32_t* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_watchdog, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_watchdog, &zero, sizeof(uint32_t));
  }
  return e;
}

cudaError_t watchdog_address(uint32_t** p) { return cudaGetSymbolAddress((void**)p, g_watchdog); }

cudaError_t takeover_count(uint32_t* value, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_takeovers, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_takeovers, &zero, sizeof(uint32_t));
  }
  return e;
}

cudaError_t launch_watchdog_selftest(uint64_t limit_ns, cudaStream_t s) {
  watchdog_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

}  // namespace mxq
