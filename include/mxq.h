/*
 * mxq.h -- C ABI of libmxq, the MX-scaled FP8 output projection ("wo_a")
 * for GB300 (sm_103a).
 *
 * The operator comes from the page "[ROCm][DSV4][Perf] Use FP8 WO_A output
 * projection" (vLLM pull request 54894), Summary items 1-2: inverse RoPE
 * fused with per-token E8M0 group quantisation of the attention output, then
 * a batched a8w8 GEMM with MX (E8M0) scales against the checkpoint's native
 * FP8 weight.  The unaligned-K linear and the load-time dequantiser come from
 * "[ROCm][DSv4.1][Perf] Dequantize the MXFP8 weight once when dot_scaled
 * cannot be used" (pull request 56560), Purpose.
 *
 * Conventions for every entry point:
 *  - Pointers are device pointers unless stated otherwise.  The caller
 *    allocates and owns every buffer; the library allocates no device memory
 *    and keeps no per-tensor state (it caches only per-device properties).
 *  - All layouts are row-major and contiguous.  "E4M3" is the OCP e4m3fn
 *    byte (bias 7, max 448, S.1111.111 = NaN, no infinity).  "E8M0" is a
 *    biased exponent byte: value 2^(byte-127), 0xFF = NaN.  BF16 is
 *    bfloat16.  Scales come one per 128 consecutive elements along the
 *    contraction axis; KG = ceil(K/128) and the last group may be partial.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  No call synchronises the host.
 *  - Argument errors are detected on the host before anything is enqueued;
 *    the call then returns the status and launches nothing.  The text of
 *    the last error of the calling thread is available from
 *    mxq_last_error().
 *  - Every device pointer must be 16-byte aligned (MXQ_ERR_ALIGN).
 *  - The device must be compute capability 10.3 (GB300); there is no
 *    fallback path (MXQ_ERR_ARCH).
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, passed as an opaque pointer so that this header needs no
 * CUDA headers. */
typedef void* mxq_stream_t;

typedef enum mxq_status {
  MXQ_OK = 0,
  MXQ_ERR_NULL = 1,        /* a required pointer is NULL */
  MXQ_ERR_SHAPE = 2,       /* a size is negative, too large or inconsistent */
  MXQ_ERR_ALIGN = 3,       /* a pointer or leading dimension is misaligned */
  MXQ_ERR_UNSUPPORTED = 4, /* a valid combination this library does not implement */
  MXQ_ERR_ARCH = 5,        /* the current device is not sm_103 */
  MXQ_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required */
  MXQ_ERR_CUDA = 7         /* a CUDA runtime/driver call failed */
} mxq_status;

/* Bits that kernels OR into a caller-provided int32 error word (err_flag).
 * Data errors never trap: the affected output is written as described at
 * each entry point and the bit is set. */
#define MXQ_DEVERR_POSITION 0x1  /* a position outside [0, max_pos) */
#define MXQ_DEVERR_SCALE 0x2     /* an FP32 scale that is not a power of two in range */
#define MXQ_DEVERR_SLOT 0x4      /* a KV-cache slot at or beyond the number of cache rows */

/* Cache element types of mxq_rope_kv_insert. */
#define MXQ_CACHE_E4M3 0 /* OCP E4M3 bytes with one per-tensor FP32 scale */
#define MXQ_CACHE_BF16 1 /* BF16 */

/* Human-readable name of a status code.  Never NULL. */
const char* mxq_status_string(int status);

/* Detail text of the last error returned to the calling thread ("" if none). */
const char* mxq_last_error(void);

/* Library ABI version: major*10000 + minor*100 + patch. */
int mxq_version(void);

/* 1 if the kernels of this library run on a device of compute capability
 * major.minor (only 10.3, GB300), else 0.  Every entry point that launches
 * work returns MXQ_ERR_ARCH on any other device. */
int mxq_arch_supported(int major, int minor);

/*
 * Fused inverse RoPE + group-128 E8M0/E4M3 quantisation of the attention
 * output.  FP8 WO_A page, Summary item 1 (the inverse rotation and the
 * per-token E8M0 group quantisation run as one kernel) and Implementation
 * (the model keeps BF16 cos/sin tables, made contiguous once at load).
 *
 *  x_bf16   [T, G, D] BF16.  Each of the T*G rows is one token's slice for
 *           one output group.
 *  pos      [T] int64 token positions.  Unused when R == 0 (may be NULL).
 *  cos_bf16, sin_bf16
 *           BF16 tables holding cos(p*theta_i) and sin(p*theta_i) of the
 *           forward rotation: row p at element offset p*cs_ld, entries
 *           i = 0..R/2-1.  cs_ld >= R/2, cs_ld % 8 == 0.  Unused when R == 0.
 *  max_pos  number of table rows.
 *  R        width of the rotated slice: the last R elements of each row,
 *           rotate-half pairs (D-R+i, D-R/2+i), i < R/2.  For c = cos[p][i],
 *           s = sin[p][i], the pair becomes
 *             y0 = fl32(x0*c + x1*s),  y1 = fl32(x1*c - x0*s)
 *           (rotation by -p*theta_i; each product is exact in fp32, so each
 *           output is one rounding).  R must be 0 or a multiple of 16 with
 *           R <= 128, and when R > 0, D % 128 == 0 (the slice lies in the
 *           last scale group).
 *  q_e4m3   [T, G, D] E4M3 codes out.
 *  q_e8m0   [T, G, ceil(D/128)] E8M0 scale bytes out.
 *  err_flag optional int32 device word; MXQ_DEVERR_POSITION is OR-ed in for a
 *           token whose position is outside [0, max_pos), and that token's
 *           codes and scale bytes are written as zeros.
 *
 * Per group (amax over the fp32 rotated values present in the group):
 *   e = smallest integer with amax <= 448 * 2^e, clamped to [-127, 127]
 *       (amax == 0 gives -127); scale byte = e + 127;
 *   code = E4M3 round-to-nearest-even, saturating, of y * 2^-e.
 * D % 16 == 0, D >= 16.  T == 0 is a no-op.  T*G*ceil(D/128) >= 2^31 returns
 * MXQ_ERR_UNSUPPORTED.
 */
int mxq_inv_rope_group_quant(const void* x_bf16, int64_t T, int32_t G, int32_t D, int32_t R,
                             const int64_t* pos, const void* cos_bf16, const void* sin_bf16,
                             int64_t cs_ld, int64_t max_pos, uint8_t* q_e4m3, uint8_t* q_e8m0,
                             int32_t* err_flag, mxq_stream_t stream);

/*
 * Size in bytes of the prepared weight-scale buffer for B weight matrices
 * of N rows and K columns.  Returns 0 for invalid sizes.
 */
size_t mxq_weight_scale_bytes(int32_t B, int32_t N, int32_t K);

/*
 * Load-time weight-scale layout transform.  FP8 WO_A page, Implementation
 * (the group-128 weight and scale layouts are checked once, at load, before
 * the FP8 path is used).  Input: w_e8m0 [B, N, ceil(K/128)] E8M0 bytes (one per weight row
 * per 128-column group).  Output: w_sf_prepared, mxq_weight_scale_bytes()
 * bytes, the layout the block-scaled GEMM reads: for each (b, group kg,
 * block of 128 rows) a 512-byte atom in which row r = 32*j + i of the block
 * owns the 32-bit word at byte offset 16*i + 4*j, holding the scale byte
 * replicated into all four bytes.  Rows are padded to a multiple of 256
 * with byte 127 (scale 1.0).  Run once after weight loading.
 */
int mxq_prepare_weight_scales(const uint8_t* w_e8m0, int32_t B, int32_t N, int32_t K,
                              uint8_t* w_sf_prepared, mxq_stream_t stream);

/* Workspace bytes mxq_bmm_a8w8 needs for these sizes (currently 0). */
size_t mxq_bmm_workspace_bytes(int64_t T, int32_t G, int32_t N, int32_t K);

/*
 * Block-scaled batched a8w8 GEMM.  FP8 WO_A page, Summary item 2 (the GEMM
 * reads the quantised activation and the weight exactly as the checkpoint
 * stores it, FP8 codes plus MX scales), with K % 128 != 0 allowed (dequantise-once page, Purpose: K = 576, 288).
 *
 *  a_e4m3    [T, G, K] activation codes; a_e8m0 [T, G, ceil(K/128)] bytes
 *            (exactly what mxq_inv_rope_group_quant writes).
 *  w_e4m3    [G, N, K] weight codes; w_sf_prepared from
 *            mxq_prepare_weight_scales(.., B=G, N, K).
 *  out_bf16  [T, G, N]:  out[t,g,n] = bf16_rne( sum_k A[t,g,k] * W[g,n,k] )
 *            with A = code * 2^(byte-127) per 128-group, likewise W; the sum
 *            is accumulated in fp32 on the tensor cores.
 *  ws        workspace of mxq_bmm_workspace_bytes() bytes (may be NULL if 0).
 * Requirements: K % 16 == 0, N % 16 == 0, K <= 65536, G >= 1.  T == 0 is a
 * no-op.  T >= 2^31, G > 65535 or N*K >= 2^40 returns MXQ_ERR_UNSUPPORTED.
 */
int mxq_bmm_a8w8(const uint8_t* a_e4m3, const uint8_t* a_e8m0, const uint8_t* w_e4m3,
                 const uint8_t* w_sf_prepared, void* out_bf16, int64_t T, int32_t G, int32_t N,
                 int32_t K, void* ws, size_t ws_bytes, mxq_stream_t stream);

/* Workspace bytes mxq_linear needs: 0 for M <= 32 (one fused launch); for
 * 32 < M <= 128 the quantised activation codes and scales plus the GEMM
 * workspace; above, mxq_wo_a_workspace_bytes(M, 1, K, N) (one launch that
 * quantises inside the GEMM). */
size_t mxq_linear_workspace_bytes(int64_t M, int32_t N, int32_t K);

/*
 * MXFP8 linear layer out[M, N] = x[M, K] * W[N, K]^T for any K % 16 == 0,
 * including K % 128 != 0, with no per-call weight dequantisation
 * (dequantise-once page, Purpose: K = 576 at TP4, 288 at TP8).  x is BF16;
 * it is quantised per row in groups of 128 exactly as
 * mxq_inv_rope_group_quant with R = 0 and multiplied as mxq_bmm_a8w8 with
 * G = 1: for M <= 32 and for M > 128 in one launch that quantises inside
 * the GEMM, in between through the workspace.  w_sf_prepared from
 * mxq_prepare_weight_scales(.., B=1, N, K).  M == 0 is a no-op.  K > 65536,
 * M >= 2^31 or N*K >= 2^40 returns MXQ_ERR_UNSUPPORTED.
 */
int mxq_linear(const void* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_sf_prepared,
               void* out_bf16, int64_t M, int32_t N, int32_t K, void* ws, size_t ws_bytes,
               mxq_stream_t stream);

/* Workspace bytes mxq_wo_a needs: 0 for T <= 32; for 32 < T <= 128, T*G*D
 * code bytes and T*G*ceil(D/128) scale bytes; for T > 128, T*G*D code
 * bytes, G*MB*ceil(D/128)*512 scale-atom bytes and G*MB*ceil(D/128)*4
 * job-counter bytes with MB = 2*ceil(T/256) (each region rounded up to 256). */
size_t mxq_wo_a_workspace_bytes(int64_t T, int32_t G, int32_t D, int32_t N);

/*
 * The whole wo_a projection in one call: mxq_inv_rope_group_quant of x
 * followed by mxq_bmm_a8w8 against W, with the same arguments, layouts,
 * rules and results (codes and scales bit-identical; the output equal to
 * the two-call sequence).  FP8 WO_A page, Summary items 1-2.
 *
 * For T <= 32 tokens (decode) it is ONE launch: the GEMM reads the BF16 x
 * and quantises each tile itself, so neither the codes nor a second launch
 * cost anything (this goes beyond the pages' two-kernel design).  For
 * 32 < T <= 128 the codes go through `ws` and two kernels run.  For T > 128
 * (prefill) it is again ONE launch: warps of the CTA-pair GEMM quantise x
 * into `ws` (codes, scale atoms, and per-job counters that the call clears
 * first) while the MMA pipeline consumes what is ready.  `ws` holds
 * mxq_wo_a_workspace_bytes(T, G, D, N) bytes, 16-byte aligned; calls that
 * may run at the same time need distinct workspaces.  err_flag as in
 * mxq_inv_rope_group_quant.  T == 0 is a no-op.  D > 65536, G > 65535,
 * T >= 2^31, N*D >= 2^40 or T*G*ceil(D/128) >= 2^31 returns
 * MXQ_ERR_UNSUPPORTED.
 */
int mxq_wo_a(const void* x_bf16, const int64_t* pos, const void* cos_bf16, const void* sin_bf16,
             int64_t cs_ld, int64_t max_pos, const uint8_t* w_e4m3, const uint8_t* w_sf_prepared,
             void* out_bf16, int64_t T, int32_t G, int32_t D, int32_t N, int32_t R,
             int32_t* err_flag, void* ws, size_t ws_bytes, mxq_stream_t stream);

/*
 * One-shot MXFP8 -> BF16 weight dequantisation.  Dequantise-once page,
 * Purpose and "Why it is worth a patch" (the BF16 weight is built once at
 * load; there it took six pointwise kernels and an FP32 intermediate, here
 * it is a single pass).  w_e4m3 [B, N, K], w_e8m0 [B, N, ceil(K/128)];
 * out_bf16[b,n,k] = bf16_rne(E4M3(code) * 2^(byte-127)) (NaN code or byte
 * 0xFF gives NaN; overflow gives +-inf).  K % 16 == 0.
 */
int mxq_dequant_bf16(const uint8_t* w_e4m3, const uint8_t* w_e8m0, void* out_bf16, int32_t B,
                     int32_t N, int32_t K, mxq_stream_t stream);

/*
 * Lossless FP32 power-of-two scales -> E8M0 bytes.  FP8 WO_A page,
 * Implementation (checkpoints may carry FP32 scales that are exact powers of
 * two; their exponent becomes the biased byte); functional-fixes page,
 * Purpose (the conversion must not rely on FP8 arithmetic, so it is done by
 * bit inspection).  s [n] float32 -> out [n] bytes:
 * 2^k with -127 <= k <= 127 gives k + 127; any other value (zero, negative,
 * not a power of two, out of range, inf, NaN) gives 0xFF and ORs
 * MXQ_DEVERR_SCALE into *err_flag (if err_flag is not NULL).
 */
int mxq_scales_f32_to_e8m0(const float* s, int64_t n, uint8_t* out, int32_t* err_flag,
                           mxq_stream_t stream);

/*
 * Forward RoPE of the query and of the new KV row, and insertion of the KV
 * row into the KV cache, in one kernel.  Functional-fixes page ("[ROCm][DSv4]
 * Functional fixes for DeepSeek V4 on MI300X/MI325X"), Purpose: the fused
 * DeepSeek V4 RoPE / KV-insert path must store the bytes of the platform's
 * FP8 encoding -- OCP E4M3, maximum 448, on the current architecture -- and
 * the cache is either BF16 or FP8 with one per-tensor scale.  The page's
 * fused kernel also normalises the query (qnorm); it states neither the norm,
 * its epsilon nor its weight, so this entry point does not normalise.
 *
 *  q_bf16     [T, H, Dq] BF16 query (H may be 0: no query).  q_out_bf16
 *             [T, H, Dq] BF16 out; it may be q_bf16 itself (in place: then
 *             only the rotated slice is read and written), but must not
 *             overlap it otherwise.
 *  kv_bf16    [T, Dk] BF16, the new KV row of each token.
 *  pos, cos_bf16, sin_bf16, cs_ld, max_pos, R
 *             as in mxq_inv_rope_group_quant, but the rotation is the
 *             forward one: for the rotate-half pairs (D-R+i, D-R/2+i) of the
 *             last R elements of every query head row and of every KV row,
 *               y0 = fl32(x0*c - x1*s),  y1 = fl32(x1*c + x0*s)
 *             (rotation by +p*theta_i; each product is exact in fp32, so
 *             each value is one rounding).  R is 0 or a multiple of 16 with
 *             R <= Dk and, when H > 0, R <= Dq.  pos/cos/sin are unused when
 *             R == 0.
 *  slot_mapping
 *             [T] int64: cache row of token t.  A negative slot writes no
 *             row (padding tokens).  Slots of different tokens must differ.
 *  kv_cache   [num_slots, Dk]: E4M3 bytes (cache_dtype MXQ_CACHE_E4M3) or
 *             BF16 (MXQ_CACHE_BF16).  Only the rows named by slot_mapping are
 *             written.
 *  kv_scale   device pointer to the per-tensor FP32 scale (E4M3 cache only;
 *             a positive finite value): the cache byte is the round-to-
 *             nearest-even, saturating (+-448) E4M3 of fl32(y / *kv_scale).
 *             The BF16 cache holds bf16_rne(y); the query output is
 *             bf16_rne(y) (elements outside the slice are copied unchanged).
 *  err_flag   optional int32 device word: MXQ_DEVERR_POSITION for a token
 *             whose position is outside [0, max_pos) (its query slices are
 *             written as zeros and its KV row is not written), and
 *             MXQ_DEVERR_SLOT for a slot >= num_slots (no row written).
 * Dq % 16 == 0 (when H > 0), Dk % 16 == 0, Dk >= 16.  T == 0 is a no-op.
 * T*H*Dq/8 + T*Dk/8 >= 2^31 returns MXQ_ERR_UNSUPPORTED.
 */
int mxq_rope_kv_insert(const void* q_bf16, void* q_out_bf16, int64_t T, int32_t H, int32_t Dq,
                       const void* kv_bf16, int32_t Dk, const int64_t* pos, const void* cos_bf16,
                       const void* sin_bf16, int64_t cs_ld, int64_t max_pos, int32_t R,
                       const int64_t* slot_mapping, void* kv_cache, int64_t num_slots,
                       int32_t cache_dtype, const float* kv_scale, int32_t* err_flag,
                       mxq_stream_t stream);

/* Size in bytes of the fixed device scratch array behind
 * mxq_linear_noalloc (4 MiB). */
#define MXQ_NOALLOC_SCRATCH_BYTES (4u * 1024u * 1024u)

/*
 * mxq_linear without a workspace argument, for callers that cannot allocate
 * device memory.  The pages have no counterpart of this entry point; it
 * exists for users of this library.
 *
 * Who needs it: a host program that links only this C library and has no
 * device allocator of its own to hand out a workspace, or a serving loop that
 * must never call cudaMalloc/cudaFree (they can synchronise the device) and
 * whose device memory was reserved up front by another component.
 *
 * Same operation, arguments, argument rules and results as mxq_linear; every
 * argument is checked before anything is enqueued.  Up to 32 rows it is
 * mxq_linear's single launch, which needs no scratch.  Above that, instead of
 * a caller-provided workspace it uses a fixed scratch array (quantiser, then
 * GEMM) that the library keeps in the device memory of every GPU it is
 * loaded on, until the process exits.  The call allocates nothing.
 *  - Limit (M > 32): the quantised activation must fit the array:
 *    round_up(M*K, 256) + round_up(M*ceil(K/128), 256) <= MXQ_NOALLOC_SCRATCH_BYTES
 *    (for example M <= 7219 rows at K = 576, 1806 at K = 2304); larger sizes return
 *    MXQ_ERR_WORKSPACE and launch nothing.
 *  - The first call on each device looks up the array's device address (a
 *    host-side runtime query, done once per device with that device current);
 *    make that first call before any stream capture.
 *  - All calls on a device share the one array, and it keeps whatever the
 *    last call left in it (every byte a call reads is first written by that
 *    same call).  Calls whose kernels overlap on the GPU -- on different
 *    streams, or from different host threads without ordering -- race on the
 *    array and give wrong results: keep them ordered, e.g. on one stream.
 */
int mxq_linear_noalloc(const void* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_sf_prepared,
                       void* out_bf16, int64_t M, int32_t N, int32_t K, mxq_stream_t stream);

/*
 * Testing aids (the pages have no counterpart), process-wide settings that
 * change no result.
 *
 * mxq_debug_set_pair_limit caps the number of CTA pairs that the many-token
 * GEMM forms launch -- mxq_bmm_a8w8, mxq_wo_a and mxq_linear above 128
 * tokens; 0 (the default) launches one pair per cluster slot that fits on
 * the device.  Every pair walks the work units with a stride of the pair
 * count, and the one-launch prefill deals its quantisation jobs by unit, so
 * any grid covers all of them.  Returns the previous cap (a negative value
 * is taken as 0).
 *
 * mxq_debug_set_lazy_pairs makes the pairs of the one-launch prefill from
 * index `from` on skip the quantisation jobs they own, as if they had not
 * started (a negative value, the default: none).  A pair that waits on a job
 * for more than 50 us quantises it itself, so a pair that is not running --
 * for example while a kernel of another stream holds SMs -- delays the
 * others instead of stalling them; this setting exercises that path.
 * Returns the previous setting.
 *
 * mxq_debug_takeovers writes to *host_value how many quantisation jobs of
 * the one-launch prefill on the current device were quantised by a waiting
 * pair instead of their owner since the last clear (host call, synchronous;
 * with clear != 0 the count is reset after reading).  0 after a call means
 * no pair ever waited 50 us for a job.  MXQ_ERR_NULL for a NULL host_value.
 */
int mxq_debug_set_pair_limit(int pairs);
int mxq_debug_set_lazy_pairs(int from);
int mxq_debug_takeovers(uint32_t* host_value, int clear);

/*
 * Watchdog word of the GEMM kernels and of the streamed query copy of
 * mxq_rope_kv_insert on the current device (host call, synchronous).  Every
 * wait inside those kernels is bounded; a wait that runs out sets a bit here
 * and the kernel returns early instead of hanging.  0 means no wait ever ran
 * out.  With clear != 0 the word is reset after reading.
 */
int mxq_watchdog_read(uint32_t* host_value, int clear);

/*
 * Self-test of the bounded-wait mechanism: enqueues one small kernel that
 * waits on a barrier nothing will ever complete.  The wait gives up after
 * limit_ns nanoseconds (1 <= limit_ns <= 2e9), the kernel sets bit 31 of the
 * watchdog word and returns normally; the context stays usable.  Used by the
 * tests to exercise the failure path without faulting the GPU.
 */
int mxq_watchdog_selftest(uint64_t limit_ns, mxq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
