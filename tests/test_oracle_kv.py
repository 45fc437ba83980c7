"""Pins of the oracle's forward RoPE and KV-cache insert (functional-fixes
page, Purpose: the fused RoPE / KV-insert path emits OCP E4M3 bytes on the
current architecture, the cache is BF16 or FP8 with a per-tensor scale, and
the RoPE region is where two implementations can round opposite ways at a
tie): a hand-worked example with ties in both encodings, the rotation
against its complex form and against the inverse rotation, single rounding,
and the encodings against torch's own conversions."""

import numpy as np
import pytest
import torch

import workloads as W
from conftest import read_sections
from oracle import mx_oracle as O


def _bits(a):
    return W.bf16_bits(torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16))


def _golden():
    sec = read_sections("rope_kv_insert_handworked.txt")
    q = np.zeros((3, 1, 128), dtype=np.float32)
    kv = np.zeros((3, 128), dtype=np.float32)
    for t, k, v in sec["q"]:
        q[int(t), 0, int(k)] = float(v)
    for t, k, v in sec["kv"]:
        kv[int(t), int(k)] = float(v)
    q_out = q.copy()
    for t, k, v in sec["q_out"]:
        q_out[int(t), 0, int(k)] = float(v)
    return sec, _bits(q), _bits(kv), _bits(q_out)


def test_rope_kv_insert_handworked_fp8():
    sec, q, kv, q_out = _golden()
    cos, sin = W.rope_cache(2, 64)
    pos = np.array([0, 1, 1])
    slots = np.array([3, 0, -1])
    cache = np.full((4, 128), 0xAA, dtype=np.uint8)
    got_q, got_cache = O.rope_kv_insert(q, kv, pos, W.bf16_bits(cos), W.bf16_bits(sin), 64, slots,
                                        cache, scale=0.5)
    want = np.full((4, 128), 0xAA, dtype=np.uint8)
    want[0] = 0
    want[3] = 0
    for r, k, c in sec["cache_fp8"]:
        want[int(r), int(k)] = int(c, 16)
    assert np.array_equal(got_cache, want)
    assert np.array_equal(got_q, q_out)


def test_rope_kv_insert_handworked_bf16():
    sec, q, kv, q_out = _golden()
    cos, sin = W.rope_cache(2, 64)
    pos = np.array([0, 1, 1])
    slots = np.array([3, 0, -1])
    cache = np.full((4, 128), 0xAAAA, dtype=np.uint16)
    got_q, got_cache = O.rope_kv_insert(q, kv, pos, W.bf16_bits(cos), W.bf16_bits(sin), 64, slots,
                                        cache)
    rows = np.zeros((4, 128), dtype=np.float32)
    for r, k, v in sec["cache_bf16"]:
        rows[int(r), int(k)] = float(v)
    want = _bits(rows)
    want[1] = 0xAAAA
    want[2] = 0xAAAA
    assert np.array_equal(got_cache, want)
    assert np.array_equal(got_q, q_out)


def test_forward_rope_position_zero_is_identity():
    x = W.bf16_normal((5, 3, 256), seed=50)
    cos, sin = W.rope_cache(4, 64)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.forward_rope_rows(xf, np.zeros(5, dtype=np.int64), W.bf16_bits(cos), W.bf16_bits(sin), 64)
    assert np.array_equal(y.view(np.uint32), xf.view(np.uint32))


def test_forward_rope_single_rounding():
    """Each rotated value is the exact x0*c - x1*s (x1*c + x0*s) rounded once to
    fp32 (BF16 products are exact in fp64 and their sum is exact there too)."""
    x = W.bf16_normal((64, 2, 128), seed=51)
    pos = W.positions_uniform(64, seed=52, max_pos=32768).numpy()
    cos, sin = W.rope_cache(32768, 64)
    cb, sb = W.bf16_bits(cos), W.bf16_bits(sin)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.forward_rope_rows(xf, pos, cb, sb, 64)
    c = O.bf16_bits_to_f32(cb[pos, :32]).astype(np.float64)[:, None, :]
    s = O.bf16_bits_to_f32(sb[pos, :32]).astype(np.float64)[:, None, :]
    x0 = xf[:, :, 64:96].astype(np.float64)
    x1 = xf[:, :, 96:128].astype(np.float64)
    assert np.array_equal(y[:, :, 64:96], (x0 * c - x1 * s).astype(np.float32))
    assert np.array_equal(y[:, :, 96:128], (x1 * c + x0 * s).astype(np.float32))
    assert np.array_equal(y[:, :, :64], xf[:, :, :64])


@pytest.mark.parametrize("R", [16, 64, 128])
def test_forward_rope_is_rotation_by_plus_angle(R):
    """Complex form (x0 + i x1) * exp(+i pos theta_i) with the exact angle, up
    to the BF16 rounding of the cache; only the last R elements move."""
    D, h = 256, R // 2
    x = W.bf16_normal((16, 2, D), seed=53 + R)
    pos = W.positions_uniform(16, seed=54 + R, max_pos=100000).numpy()
    cos, sin = W.rope_cache(100000, R)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.forward_rope_rows(xf, pos, W.bf16_bits(cos), W.bf16_bits(sin), R).astype(np.float64)
    theta = 10000.0 ** (-2.0 * np.arange(h) / R)
    ang = pos[:, None, None].astype(np.float64) * theta
    x0 = xf[:, :, D - R:D - h].astype(np.float64)
    x1 = xf[:, :, D - h:].astype(np.float64)
    z = (x0 + 1j * x1) * np.exp(1j * ang)
    bound = 2.0 ** -8 * 2 * (np.abs(x0) + np.abs(x1)) + 1e-6
    assert np.all(np.abs(y[:, :, D - R:D - h] - z.real) <= bound)
    assert np.all(np.abs(y[:, :, D - h:] - z.imag) <= bound)
    assert np.array_equal(y[:, :, :D - R], xf[:, :, :D - R].astype(np.float64))


def test_inverse_of_forward_round_trip():
    x = W.bf16_normal((16, 4, 192), seed=55)
    pos = W.positions_uniform(16, seed=56, max_pos=32768).numpy()
    cos, sin = W.rope_cache(32768, 64)
    cb, sb = W.bf16_bits(cos), W.bf16_bits(sin)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.forward_rope_rows(xf, pos, cb, sb, 64)
    back = O.inverse_rope_rows(y, pos, cb, sb, 64).astype(np.float64)
    c = O.bf16_bits_to_f32(cb[pos, :32]).astype(np.float64)[:, None, :]
    s = O.bf16_bits_to_f32(sb[pos, :32]).astype(np.float64)[:, None, :]
    x0, x1 = xf[:, :, 128:160], xf[:, :, 160:192]
    bound = (np.abs(c * c + s * s - 1.0) + 2.0 ** -21) * (np.abs(x0) + np.abs(x1)) + 1e-30
    assert np.all(np.abs(back[:, :, 128:160] - x0) <= bound)
    assert np.all(np.abs(back[:, :, 160:192] - x1) <= bound)
    assert np.array_equal(back[:, :, :128], xf[:, :, :128])


def _random_case(seed, T=24, H=3, Dq=192, Dk=256, R=64, max_pos=5000):
    q = W.bf16_normal((T, H, Dq), seed=seed)
    kv = W.bf16_normal((T, Dk), seed=seed + 1, std=4.0)
    pos = W.positions_uniform(T, seed=seed + 2, max_pos=max_pos).numpy()
    cos, sin = W.rope_cache(max_pos, R)
    return W.bf16_bits(q), W.bf16_bits(kv), pos, W.bf16_bits(cos), W.bf16_bits(sin)


@pytest.mark.parametrize("scale", [0.5, 0.0371, 3.0])
def test_fp8_cache_rows_match_torch(scale):
    """Cache rows = torch's float32 -> float8_e4m3fn (RNE) of fl32(rope(kv) / scale),
    rope(kv) from the forward rotation; rows written at their slots only."""
    q, kv, pos, cb, sb = _random_case(60)
    T, Dk = kv.shape
    slots = np.arange(T)[::-1] * 2
    slots[5] = -1
    cache = np.full((2 * T, Dk), 0x5A, dtype=np.uint8)
    _, out = O.rope_kv_insert(q, kv, pos, cb, sb, 64, slots, cache, scale=scale)
    k = O.forward_rope_rows(O.bf16_bits_to_f32(kv)[:, None, :], pos, cb, sb, 64)[:, 0, :]
    v = torch.from_numpy(k) / torch.tensor(scale, dtype=torch.float32)
    assert float(v.abs().max()) < 448.0  # torch gives NaN above the range, the cache saturates
    want = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t in range(T):
        if slots[t] >= 0:
            assert np.array_equal(out[slots[t]], want[t]), t
    untouched = np.setdiff1d(np.arange(2 * T), slots[slots >= 0])
    assert (out[untouched] == 0x5A).all()


def test_bf16_outputs_match_torch():
    """q_out and the BF16 cache rows = torch's float32 -> bfloat16 of the
    rotated fp32 values."""
    q, kv, pos, cb, sb = _random_case(70)
    T, Dk = kv.shape
    slots = np.arange(T)
    cache = np.zeros((T, Dk), dtype=np.uint16)
    q_out, out = O.rope_kv_insert(q, kv, pos, cb, sb, 64, slots, cache)
    yq = O.forward_rope_rows(O.bf16_bits_to_f32(q), pos, cb, sb, 64)
    yk = O.forward_rope_rows(O.bf16_bits_to_f32(kv)[:, None, :], pos, cb, sb, 64)[:, 0, :]
    assert np.array_equal(q_out, W.bf16_bits(torch.from_numpy(yq).to(torch.bfloat16)))
    assert np.array_equal(out, W.bf16_bits(torch.from_numpy(yk).to(torch.bfloat16)))


def test_no_rotation_passes_values_through():
    """R = 0: the query is copied bit for bit and the cache holds E4M3(kv / scale)."""
    q, kv, pos, cb, sb = _random_case(80)
    T, Dk = kv.shape
    q_out, out = O.rope_kv_insert(q, kv, pos, cb, sb, 0, np.arange(T),
                                  np.zeros((T, Dk), dtype=np.uint8), scale=2.0)
    assert np.array_equal(q_out, q)
    v = torch.from_numpy(O.bf16_bits_to_f32(kv)) / 2.0
    assert np.array_equal(out, v.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_fp8_scale_division_rounds_once_in_fp32():
    """The FP8 cache code is E4M3 of the fp32 quotient: with kv = 1.0 and the
    scale 0x3F579436 (0.84210526943...), 1 / scale is 1.1875 - 8.8e-9 exactly,
    but its fp32 rounding is 1.1875, the midpoint of 1.125 (mantissa 1) and
    1.25 (mantissa 2): the tie goes to the even mantissa, 1.25, code 0x3A
    (dividing in higher precision would give 1.125, code 0x39)."""
    scale = float(np.uint32(0x3F579436).view(np.float32))
    kv = _bits(np.array([[1.0] + [0.0] * 15], dtype=np.float32))
    q = _bits(np.zeros((1, 1, 16), dtype=np.float32))
    cos, sin = W.rope_cache(1, 2)
    _, out = O.rope_kv_insert(q, kv, np.array([0]), W.bf16_bits(cos), W.bf16_bits(sin), 0,
                              np.array([0]), np.zeros((1, 16), dtype=np.uint8), scale=scale)
    assert out[0, 0] == 0x3A
    assert (out[0, 1:] == 0).all()
