"""Plain, slow CPU oracle for the MX-scaled FP8 ``wo_a`` path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code, table or helper with the
CUDA library; the two meet only on the seeded inputs from ``workloads``.

What it computes, and where each step comes from:

* Page "[ROCm][DSV4][Perf] Use FP8 WO_A output projection", Summary items 1-2:
  the attention output is un-rotated (inverse RoPE) and quantised per token
  in 128-wide groups with one E8M0 scale each, in one pass; a batched a8w8
  GEMM then multiplies it by the FP8 weight as stored in the checkpoint,
  codes plus MX scales.  Implementation section: scales come either as E8M0
  bytes or as FP32 exact powers of two whose exponent becomes the byte; the
  layouts are group-128; the cos/sin tables are BF16.
* Page "[ROCm][DSv4] Functional fixes for DeepSeek V4 on MI300X/MI325X",
  Purpose: OCP E4M3 encoding (max 448) on the current architecture, scale
  conversion by bit manipulation rather than FP8 arithmetic.
* Page "[ROCm][DSv4.1][Perf] Dequantize the MXFP8 weight once when
  dot_scaled cannot be used", Purpose and "Why it is worth a patch": the
  BF16 copy of an MXFP8 weight is each decoded E4M3 value times
  2^(scale byte - 127), rounded once to BF16; the unaligned shapes are
  K = 576 and 288.

Readings taken where the pages are silent:

* Scale rule: e = ceil(log2(amax / 448)), i.e. the smallest integer e with
  amax <= 448 * 2^e, evaluated exactly (no floating log2 or division);
  amax == 0 gives e = -127; e is clamped to [-127, 127]; byte = e + 127.
* E4M3 encode: round to nearest, ties to the even code, saturate at +-448,
  the sign of zero kept.
* Inverse RoPE: rotate-half pairs (D-R+i, D-R+R/2+i) of the last R elements
  of each row, angle -pos*theta_i, with the tables holding the forward
  cos(pos*theta_i), sin(pos*theta_i) in BF16.  Each output is one fp32
  rounding of x0*c + x1*s (the BF16 x BF16 products are exact in fp32), and
  the rotated values stay fp32 (they are not rounded to BF16) before
  quantisation.
* A partial last group (K % 128 != 0) takes its amax over the elements that
  exist.
* GEMM reference: exact products summed in fp64; GPU results are checked by
  |y - y_ref| <= 1 bf16 ulp(y_ref) + 1e-5 * sum_k |a_k w_k|.

Parity is pinned by tests/test_oracle_*.py (hand-worked examples, library
routines for the encodings, exact rational brute force, invariants).
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

E4M3_MAX = 448.0
GROUP = 128


# --------------------------------------------------------------------------
# OCP E4M3 (e4m3fn) code table.
# Functional-fixes page, Purpose: the current architecture uses the OCP
# encoding with maximum 448 (FNUZ, max 224, is the other one and is not used).
# --------------------------------------------------------------------------
def e4m3_decode_one(code: int) -> float:
    """Value of one OCP E4M3 byte: sign, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent field 0 is subnormal (M * 2^-9); S.1111.111 is NaN; there
    is no infinity."""
    s = (code >> 7) & 1
    E = (code >> 3) & 0xF
    M = code & 0x7
    if E == 0xF and M == 0x7:
        return math.nan
    if E == 0:
        mag = M * 2.0 ** -9
    else:
        mag = (1.0 + M / 8.0) * 2.0 ** (E - 7)
    return -mag if s else mag


E4M3_TABLE = np.array([e4m3_decode_one(c) for c in range(256)], dtype=np.float64)
# Non-negative finite codes 0x00..0x7E are ordered by value.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = E4M3_TABLE[:0x7F]


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Table decode of an array of E4M3 bytes to float64 (NaN for 0x7F/0xFF)."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8).astype(np.int64)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code to each float64 value, by search in the value table.

    Ties go to the code with an even mantissa (even code), magnitudes above
    448 saturate to 0x7E/0xFE, NaN gives 0x7F, and the sign bit is kept on
    zero results."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    neg = np.signbit(v)
    hi = np.searchsorted(_POS_VALUES, a, side="left")  # first table value >= a
    hi = np.clip(hi, 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (_POS_CODES[lo] % 2 == 0))
    code = np.where(pick_lo, _POS_CODES[lo], _POS_CODES[hi])
    code = np.where(a >= E4M3_MAX, 0x7E, code)  # saturate
    code = code | np.where(neg, 0x80, 0)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# E8M0 scale exponent for one group.
# --------------------------------------------------------------------------
def e8m0_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127];
    amax == 0 gives -127.

    frexp gives amax = m * 2^E exactly with m in [0.5, 1).  Then
    amax * 2^-(E-9) = m * 512 lies in [256, 512): it is <= 448 exactly when
    m <= 0.875, and e = E - 10 would give m * 1024 >= 512 > 448.  So
    e = E - 9 if m <= 0.875, else E - 8."""
    amax = np.asarray(amax, dtype=np.float64)
    m, E = np.frexp(amax)
    e = E.astype(np.int64) - 9 + (m > 0.875).astype(np.int64)
    e = np.where(amax == 0.0, -127, e)
    return np.clip(e, -127, 127)


# --------------------------------------------------------------------------
# Inverse RoPE (fp32, fixed evaluation order).
# FP8 WO_A page, Summary item 1 (the inverse rotation runs inside the
# quantisation kernel) and Implementation (BF16 cos/sin tables kept by the
# model).
# --------------------------------------------------------------------------
def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns (uint16) to float32; exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def inverse_rope_rows(x_f32: np.ndarray, pos: np.ndarray, cos_bits: np.ndarray,
                      sin_bits: np.ndarray, R: int) -> np.ndarray:
    """Un-rotate the last R elements of each row.

    x_f32: [T, G, D] float32 (widened BF16); pos: [T] int; cos_bits, sin_bits:
    [max_pos, >= R/2] BF16 bit patterns holding cos(pos*theta_i), sin(pos*theta_i).
    For i < R/2, j0 = D-R+i, j1 = j0+R/2, c = cos[pos][i], s = sin[pos][i]:
        y[j0] = fl32(fl32(x[j0]*c) + fl32(x[j1]*s))
        y[j1] = fl32(fl32(x[j1]*c) - fl32(x[j0]*s))
    which is a rotation by -pos*theta_i.  Elements before D-R pass through."""
    y = np.array(x_f32, dtype=np.float32, copy=True)
    if R == 0:
        return y
    T, G, D = y.shape
    half = R // 2
    for t in range(T):
        p = int(pos[t])
        c = bf16_bits_to_f32(cos_bits[p, :half])  # [half]
        s = bf16_bits_to_f32(sin_bits[p, :half])
        x0 = x_f32[t, :, D - R:D - half].astype(np.float32)  # [G, half]
        x1 = x_f32[t, :, D - half:D].astype(np.float32)
        y[t, :, D - R:D - half] = (x0 * c) + (x1 * s)  # numpy float32: IEEE RN, no FMA
        y[t, :, D - half:D] = (x1 * c) - (x0 * s)
    return y


def group_quant_rows(y: np.ndarray):
    """Per-row group-128 quantisation of float32 rows [..., D].

    For each group (the last one partial when D % 128 != 0): amax over the
    group, e = e8m0_exponent(amax), code = E4M3_RNE_satfinite(y * 2^-e),
    scale byte = e + 127.  Returns (codes uint8 [..., D],
    scales uint8 [..., ceil(D/128)])."""
    y = np.asarray(y, dtype=np.float32)
    D = y.shape[-1]
    KG = (D + GROUP - 1) // GROUP
    codes = np.empty(y.shape, dtype=np.uint8)
    scales = np.empty(y.shape[:-1] + (KG,), dtype=np.uint8)
    for kg in range(KG):
        blk = y[..., kg * GROUP:min(D, (kg + 1) * GROUP)].astype(np.float64)
        amax = np.max(np.abs(blk), axis=-1)
        e = e8m0_exponent(amax)
        v = np.ldexp(blk, -e[..., None])  # exact power-of-two scaling in fp64
        codes[..., kg * GROUP:min(D, (kg + 1) * GROUP)] = e4m3_encode(v)
        scales[..., kg] = (e + 127).astype(np.uint8)
    return codes, scales


def inv_rope_group_quant(x_bits: np.ndarray, pos: np.ndarray, cos_bits: np.ndarray,
                         sin_bits: np.ndarray, R: int):
    """Oracle of mxq_inv_rope_group_quant.

    x_bits: BF16 bit patterns [T, G, D] (uint16).  Returns (codes [T,G,D],
    scales [T,G,ceil(D/128)]), both uint8."""
    x = bf16_bits_to_f32(x_bits)
    y = inverse_rope_rows(x, pos, cos_bits, sin_bits, R)
    return group_quant_rows(y)


# --------------------------------------------------------------------------
# Dequantisation to BF16.
# Dequantize-once page, Purpose: the load-time BF16 weight; its Test Result
# profile shows the value built as exp2 of the integer scale exponent times
# the decoded code.
# --------------------------------------------------------------------------
def bf16_rne_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to BF16 (round to nearest, ties to even), with
    subnormals (quantum 2^-133) and overflow to infinity.  NaN -> 0x7FC0."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    m, E = np.frexp(a)  # a = m * 2^E, m in [0.5, 1)
    # 8 significant bits: quantum 2^(E-8) for normal values, 2^-133 below 2^-126
    q = np.maximum(E.astype(np.int64) - 8, -133)
    n = np.rint(np.ldexp(a, -q))  # exact scaling, then round half to even
    r = np.ldexp(n, q)
    r = np.where(a == 0.0, 0.0, r)
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    r = np.where(np.isinf(a), np.inf, r)
    bits = (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = bits | np.where(np.signbit(v), np.uint16(0x8000), np.uint16(0))
    bits = np.where(np.isnan(v), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def e8m0_value(sc: np.ndarray) -> np.ndarray:
    """2^(byte - 127) in float64; byte 0xFF is NaN."""
    sc = np.asarray(sc, dtype=np.int64)
    val = np.ldexp(np.ones(sc.shape), sc - 127)
    return np.where(sc == 255, np.nan, val)


def mx_values(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Exact float64 values code * 2^(scale-127), scales per 128-group along
    the last axis.  codes [..., K], scales [..., ceil(K/128)]."""
    K = codes.shape[-1]
    sc_full = np.repeat(np.asarray(scales), GROUP, axis=-1)[..., :K]
    return e4m3_decode(codes) * e8m0_value(sc_full)


def dequant_bf16(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Oracle of mxq_dequant_bf16: BF16 bits of RNE(code * 2^(scale-127))."""
    return bf16_rne_bits(mx_values(codes, scales))


# --------------------------------------------------------------------------
# Block-scaled batched GEMM.
# FP8 WO_A page, Summary item 2: batched a8w8 GEMM of the quantised
# activation against the native FP8 weight with MX scales.
# --------------------------------------------------------------------------
def bmm_a8w8_ref(a_codes, a_scales, w_codes, w_scales):
    """y_ref[t,g,n] = sum_k A[t,g,k] * W[g,n,k] in float64, and
    S[t,g,n] = sum_k |A[t,g,k] * W[g,n,k]|, with A and W the exact MX values.

    a_codes [T,G,K], a_scales [T,G,KG], w_codes [G,N,K], w_scales [G,N,KG]."""
    A = mx_values(a_codes, a_scales)  # [T,G,K]
    W = mx_values(w_codes, w_scales)  # [G,N,K]
    T, G, K = A.shape
    N = W.shape[1]
    y = np.empty((T, G, N), dtype=np.float64)
    S = np.empty((T, G, N), dtype=np.float64)
    for g in range(G):
        y[:, g, :] = A[:, g, :] @ W[g].T
        S[:, g, :] = np.abs(A[:, g, :]) @ np.abs(W[g]).T
    return y, S


def linear_ref(x_bits, w_codes, w_scales):
    """Oracle of mxq_linear: quantise x [M,K] per token in groups of 128
    (no RoPE), then the block-scaled GEMM with one group.
    Returns (y_ref [M,N], S [M,N], a_codes, a_scales)."""
    x = bf16_bits_to_f32(x_bits)  # [M,K]
    a_codes, a_scales = group_quant_rows(x)
    y, S = bmm_a8w8_ref(a_codes[:, None, :], a_scales[:, None, :],
                        w_codes[None], w_scales[None])
    return y[:, 0, :], S[:, 0, :], a_codes, a_scales


def bf16_ulp(y_ref: np.ndarray) -> np.ndarray:
    """One BF16 ulp at y_ref: 2^(max(floor(log2|y|), -126) - 7); 2^-133 at 0."""
    a = np.abs(np.asarray(y_ref, dtype=np.float64))
    m, E = np.frexp(a)  # a = m*2^E, floor(log2 a) = E-1
    ex = np.maximum(E.astype(np.int64) - 1, -126) - 7
    return np.where(a == 0.0, 2.0 ** -133, np.ldexp(np.ones(a.shape), ex))


def gemm_tolerance(y_ref, S):
    """Allowed |y - y_ref|: 1 bf16 ulp of y_ref plus 1e-5 * sum_k |a_k w_k|."""
    return bf16_ulp(y_ref) + 1e-5 * np.asarray(S, dtype=np.float64)


# --------------------------------------------------------------------------
# FP32 power-of-two scales -> E8M0 bytes.
# FP8 WO_A page, Implementation: an FP32 scale that is an exact positive power
# of two carries no information beyond its exponent, so it maps losslessly to
# the biased byte; functional-fixes page: no FP8 arithmetic in the conversion.
# --------------------------------------------------------------------------
def scales_f32_to_e8m0(s: np.ndarray):
    """Returns (bytes uint8, ok bool).  A value is accepted when it is a
    positive finite power of two 2^k with -127 <= k <= 127; the byte is k+127.
    Anything else gives byte 0xFF and ok=False."""
    s = np.asarray(s, dtype=np.float32).astype(np.float64)
    m, E = np.frexp(s)
    k = E.astype(np.int64) - 1
    ok = np.isfinite(s) & (s > 0) & (m == 0.5) & (k >= -127) & (k <= 127)
    out = np.where(ok, k + 127, 255).astype(np.uint8)
    return out, ok


# --------------------------------------------------------------------------
# Forward RoPE and insertion of the new KV row into an FP8 or BF16 cache.
# Functional-fixes page, Purpose: the fused DeepSeek V4 RoPE / KV-insert path
# must emit the bytes of the platform's FP8 encoding, OCP E4M3 (max 448) on
# the current architecture; the cache is checked either as BF16 or as FP8
# with a per-tensor scale ("full-cache per-tensor FP8"), and the RoPE region
# is where a kernel and a reference can round opposite ways at ties.
# Readings: the rotation is the forward one of the wo_a cache (+pos*theta_i,
# rotate-half pairs of the last R elements of a row); the rotated values stay
# fp32 and are rounded once, to BF16 (query, BF16 cache) or, divided by the
# per-tensor scale in fp32, to E4M3 (FP8 cache); a negative slot skips the
# token's cache row.
# --------------------------------------------------------------------------
def forward_rope_rows(x_f32: np.ndarray, pos: np.ndarray, cos_bits: np.ndarray,
                      sin_bits: np.ndarray, R: int) -> np.ndarray:
    """Rotate the last R elements of each row by +pos*theta_i.

    x_f32: [T, H, D] float32 (widened BF16).  For i < R/2, j0 = D-R+i,
    j1 = j0+R/2, c = cos[pos][i], s = sin[pos][i]:
        y[j0] = fl32(fl32(x[j0]*c) - fl32(x[j1]*s))
        y[j1] = fl32(fl32(x[j1]*c) + fl32(x[j0]*s))
    (with a = x[j0], b = x[j1], cs = c, sn = s below).
    Elements before D-R pass through."""
    y = np.array(x_f32, dtype=np.float32, copy=True)
    if R == 0:
        return y
    T, H, D = y.shape
    h = R // 2
    for t in range(T):
        row = int(pos[t])
        cs = bf16_bits_to_f32(cos_bits[row, :h])
        sn = bf16_bits_to_f32(sin_bits[row, :h])
        a = x_f32[t, :, D - R:D - h].astype(np.float32)
        b = x_f32[t, :, D - h:D].astype(np.float32)
        y[t, :, D - R:D - h] = (a * cs) - (b * sn)  # numpy float32: IEEE RN, no FMA
        y[t, :, D - h:D] = (b * cs) + (a * sn)
    return y


def rope_kv_insert(q_bits, kv_bits, pos, cos_bits, sin_bits, R, slots, cache, scale=None):
    """Oracle of mxq_rope_kv_insert.

    q_bits [T, H, Dq] and kv_bits [T, Dk]: BF16 bit patterns; pos [T] valid
    table rows; slots [T] cache rows (negative: no write).  cache: the cache
    before the call, [num_slots, Dk], uint8 E4M3 codes when `scale` is given,
    else uint16 BF16 bits.  Returns (q_out bits [T, H, Dq], the cache after the
    call).  q_out = BF16_RNE(forward RoPE of q); the cache row of token t is
    E4M3_RNE_satfinite(fl32(rope(kv) / scale)) or BF16_RNE(rope(kv)), written
    in token order."""
    q = bf16_bits_to_f32(q_bits)
    kv = bf16_bits_to_f32(kv_bits)[:, None, :]
    q_out = bf16_rne_bits(forward_rope_rows(q, pos, cos_bits, sin_bits, R).astype(np.float64))
    k = forward_rope_rows(kv, pos, cos_bits, sin_bits, R)[:, 0, :]
    if scale is None:
        rows = bf16_rne_bits(k.astype(np.float64))
    else:
        v = k / np.float32(scale)  # one IEEE fp32 division
        rows = e4m3_encode(v.astype(np.float64))
    out = np.array(cache, copy=True)
    for t in range(len(slots)):
        if int(slots[t]) >= 0:
            out[int(slots[t])] = rows[t]
    return q_out, out


# --------------------------------------------------------------------------
# Exact rational helpers for brute-force pins on tiny shapes.
# --------------------------------------------------------------------------
def e4m3_fraction(code: int) -> Fraction:
    """Exact rational value of a finite E4M3 code."""
    s = (code >> 7) & 1
    E = (code >> 3) & 0xF
    M = code & 0x7
    if E == 0:
        mag = Fraction(M, 2 ** 9)
    else:
        mag = Fraction(8 + M, 8) * (Fraction(2) ** (E - 7))
    return -mag if s else mag


def dot_exact(a_codes, a_scales, w_codes, w_scales) -> Fraction:
    """Exact sum_k A_k W_k for one (row, weight-row) pair, as a Fraction."""
    total = Fraction(0)
    for k in range(len(a_codes)):
        sa = Fraction(2) ** (int(a_scales[k // GROUP]) - 127)
        sw = Fraction(2) ** (int(w_scales[k // GROUP]) - 127)
        total += e4m3_fraction(int(a_codes[k])) * sa * e4m3_fraction(int(w_codes[k])) * sw
    return total
