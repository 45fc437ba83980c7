"""Pins of the oracle's inverse RoPE, group quantisation and block-scaled
GEMM: the hand-worked two-token example, exact rational brute force,
invariants (rotation round trip, position 0, quantisation error bound) and
special cases (all-ones / one-hot weights, zero-padded K tail)."""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W
from conftest import read_sections
from oracle import mx_oracle as O


def _golden_2tok():
    sec = read_sections("wo_a_2token_handworked.txt")
    x = np.zeros((2, 1, 128), dtype=np.float32)
    for t, k, v in sec["x"]:
        x[int(t), 0, int(k)] = float(v)
    x_bits = W.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    pos = np.array([int(p) for _, p in sec["pos"]], dtype=np.int64)
    codes = np.zeros((2, 1, 128), dtype=np.uint8)
    for t, k, c in sec["codes"]:
        codes[int(t), 0, int(k)] = int(c, 16)
    scales = np.zeros((2, 1, 1), dtype=np.uint8)
    for t, b in sec["scales"]:
        scales[int(t), 0, 0] = int(b)
    return sec, x_bits, pos, codes, scales


def test_rope_cache_handworked_entries():
    cos, sin = W.rope_cache(2, 64)
    c, s = cos.float().numpy(), sin.float().numpy()
    assert (c[0] == 1.0).all() and (s[0] == 0.0).all()
    assert c[1, 0] == 0.5390625 and s[1, 0] == 0.83984375
    assert c[1, 6] == 0.984375 and s[1, 6] == 0.1767578125


def test_two_token_handworked_quant():
    _, x_bits, pos, codes, scales = _golden_2tok()
    cos, sin = W.rope_cache(2, 64)
    q, sc = O.inv_rope_group_quant(x_bits, pos, W.bf16_bits(cos), W.bf16_bits(sin), 64)
    assert np.array_equal(sc, scales)
    assert np.array_equal(q, codes), np.argwhere(q != codes)


def test_two_token_handworked_gemm():
    sec, x_bits, pos, codes, scales = _golden_2tok()
    w = np.zeros((1, 3, 128), dtype=np.uint8)
    w[0, 0, :] = 0x38
    w[0, 1, 64] = 0x40
    w[0, 2, 5] = 0x38
    w[0, 2, 96] = 0xB8
    ws = np.zeros((1, 3, 1), dtype=np.uint8)
    for n, b in sec["w_scales"]:
        ws[0, int(n), 0] = int(b)
    y, S = O.bmm_a8w8_ref(codes, scales, w, ws)
    for t, n, v, bits in sec["y"]:
        assert y[int(t), 0, int(n)] == float(v)
        assert int(O.bf16_rne_bits(np.array([y[int(t), 0, int(n)]]))[0]) == int(bits, 16)


def test_inverse_rope_position_zero_is_identity():
    x = W.bf16_normal((5, 3, 256), seed=1)
    cos, sin = W.rope_cache(4, 64)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.inverse_rope_rows(xf, np.zeros(5, dtype=np.int64), W.bf16_bits(cos), W.bf16_bits(sin), 64)
    assert np.array_equal(y.view(np.uint32), xf.view(np.uint32))


def test_inverse_rope_single_rounding():
    """Each rotated value is the exact x0*c + x1*s rounded once to fp32."""
    x = W.bf16_normal((64, 2, 128), seed=2)
    pos = W.positions_uniform(64, seed=3, max_pos=32768).numpy()
    cos, sin = W.rope_cache(32768, 64)
    cb, sb = W.bf16_bits(cos), W.bf16_bits(sin)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.inverse_rope_rows(xf, pos, cb, sb, 64)
    c = O.bf16_bits_to_f32(cb[pos, :32]).astype(np.float64)[:, None, :]
    s = O.bf16_bits_to_f32(sb[pos, :32]).astype(np.float64)[:, None, :]
    x0 = xf[:, :, 64:96].astype(np.float64)
    x1 = xf[:, :, 96:128].astype(np.float64)
    assert np.array_equal(y[:, :, 64:96], (x0 * c + x1 * s).astype(np.float32))
    assert np.array_equal(y[:, :, 96:128], (x1 * c - x0 * s).astype(np.float32))
    assert np.array_equal(y[:, :, :64], xf[:, :, :64])


def test_inverse_rope_is_rotation_by_minus_angle():
    """Complex form: (x0 + i x1) * exp(-i pos theta) with the exact angle, up to
    the BF16 rounding of the cache."""
    x = W.bf16_normal((32, 1, 64), seed=4)
    pos = W.positions_uniform(32, seed=5, max_pos=4096).numpy()
    cos, sin = W.rope_cache(4096, 64)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.inverse_rope_rows(xf, pos, W.bf16_bits(cos), W.bf16_bits(sin), 64).astype(np.float64)
    theta = 10000.0 ** (-2.0 * np.arange(32) / 64)
    ang = pos[:, None].astype(np.float64) * theta[None, :]
    z = (xf[:, 0, :32] + 1j * xf[:, 0, 32:]) * np.exp(-1j * ang)
    bound = 2.0 ** -8 * 2 * (np.abs(xf[:, 0, :32]) + np.abs(xf[:, 0, 32:])) + 1e-6
    assert np.all(np.abs(y[:, 0, :32] - z.real) <= bound)
    assert np.all(np.abs(y[:, 0, 32:] - z.imag) <= bound)


@pytest.mark.parametrize("R", [16, 128])
def test_inverse_rope_other_widths(R):
    """The narrowest and widest rotated slices: only the last R elements move,
    as pairs (D-R+i, D-R/2+i) rotated by -pos*theta_i, theta_i = 10000^(-2i/R)."""
    D, h = 256, R // 2
    x = W.bf16_normal((16, 2, D), seed=40 + R)
    pos = W.positions_uniform(16, seed=41 + R, max_pos=4096).numpy()
    cos, sin = W.rope_cache(4096, R)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.inverse_rope_rows(xf, pos, W.bf16_bits(cos), W.bf16_bits(sin), R).astype(np.float64)
    theta = 10000.0 ** (-2.0 * np.arange(h) / R)
    ang = pos[:, None, None].astype(np.float64) * theta
    x0 = xf[:, :, D - R:D - h].astype(np.float64)
    x1 = xf[:, :, D - h:].astype(np.float64)
    z = (x0 + 1j * x1) * np.exp(-1j * ang)
    bound = 2.0 ** -8 * 2 * (np.abs(x0) + np.abs(x1)) + 1e-6
    assert np.all(np.abs(y[:, :, D - R:D - h] - z.real) <= bound)
    assert np.all(np.abs(y[:, :, D - h:] - z.imag) <= bound)
    assert np.array_equal(y[:, :, :D - R], xf[:, :, :D - R].astype(np.float64))


def test_rope_of_inverse_rope_round_trip():
    x = W.bf16_normal((16, 4, 192), seed=6)
    pos = W.positions_uniform(16, seed=7, max_pos=32768).numpy()
    cos, sin = W.rope_cache(32768, 64)
    cb, sb = W.bf16_bits(cos), W.bf16_bits(sin)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x))
    y = O.inverse_rope_rows(xf, pos, cb, sb, 64).astype(np.float64)
    c = O.bf16_bits_to_f32(cb[pos, :32]).astype(np.float64)[:, None, :]
    s = O.bf16_bits_to_f32(sb[pos, :32]).astype(np.float64)[:, None, :]
    y0, y1 = y[:, :, 128:160], y[:, :, 160:192]
    r0 = y0 * c - y1 * s  # forward rotation
    r1 = y1 * c + y0 * s
    x0, x1 = xf[:, :, 128:160], xf[:, :, 160:192]
    bound = (np.abs(c * c + s * s - 1.0) + 2.0 ** -22) * (np.abs(x0) + np.abs(x1)) + 1e-30
    assert np.all(np.abs(r0 - x0) <= bound)
    assert np.all(np.abs(r1 - x1) <= bound)


def test_quant_error_bound_and_scale_range():
    x = W.bf16_normal((8, 2, 512), seed=8, outlier_frac=0.01)
    xf = O.bf16_bits_to_f32(W.bf16_bits(x)).astype(np.float64)
    codes, scales = O.group_quant_rows(xf.astype(np.float32))
    xhat = O.mx_values(codes, scales)
    e = np.repeat(scales.astype(np.int64) - 127, 128, axis=-1)
    a = np.abs(xf)
    normal = a >= np.ldexp(1.0, e - 6)
    lg = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    bound = np.where(normal, np.exp2(lg - 4), np.ldexp(1.0, e - 10))
    assert np.all(np.abs(xf - xhat) <= bound)
    # each group's largest code magnitude lies in [224, 448] (224.x may round down to 224)
    mags = np.abs(O.e4m3_decode(codes)).reshape(8, 2, 4, 128).max(axis=-1)
    assert np.all((mags >= 224) & (mags <= 448))


def test_partial_last_group_uses_only_present_elements():
    x = np.zeros((1, 1, 288), dtype=np.float32)
    x[0, 0, :256] = 100.0
    x[0, 0, 256:] = 0.25
    codes, scales = O.group_quant_rows(x)
    assert list(scales[0, 0]) == [127 - 2, 127 - 2, 127 - 10]  # 100 -> e=-2, 0.25 -> e=-10
    assert (codes[0, 0, 256:] == O.e4m3_encode(np.array([0.25 * 1024]))[0]).all()


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    return c


def test_gemm_exact_rational_brute_force():
    rng = np.random.Generator(np.random.PCG64(21))
    T, G, N, K = 3, 2, 4, 160  # partial second group
    KG = 2
    a = _rand_codes(rng, (T, G, K))
    sa = rng.integers(110, 140, size=(T, G, KG), dtype=np.uint8)
    w = _rand_codes(rng, (G, N, K))
    sw = rng.integers(110, 140, size=(G, N, KG), dtype=np.uint8)
    y, S = O.bmm_a8w8_ref(a, sa, w, sw)
    for t in range(T):
        for g in range(G):
            for n in range(N):
                ex = O.dot_exact(a[t, g], sa[t, g], w[g, n], sw[g, n])
                # fp64 accumulation of exact products: error <= K * 2^-53 * S
                assert abs(Fraction(y[t, g, n]) - ex) <= Fraction(K) * Fraction(2) ** -53 * Fraction(S[t, g, n])
                # S is the sum of the magnitudes of the same exact products
                ex_abs = sum(abs(O.dot_exact(a[t, g, k:k + 1], sa[t, g, k // 128:], w[g, n, k:k + 1],
                                             sw[g, n, k // 128:])) for k in range(K))
                assert abs(Fraction(S[t, g, n]) - ex_abs) <= Fraction(K) * Fraction(2) ** -53 * ex_abs


def test_gemm_special_cases():
    rng = np.random.Generator(np.random.PCG64(22))
    T, G, K = 4, 2, 256
    a = _rand_codes(rng, (T, G, K))
    sa = rng.integers(115, 135, size=(T, G, 2), dtype=np.uint8)
    A = O.mx_values(a, sa)
    w = np.zeros((G, K + 1, K), dtype=np.uint8)
    w[:, 0, :] = 0x38  # ones
    for k in range(K):
        w[:, k + 1, k] = 0x38  # one-hot
    sw = np.full((G, K + 1, 2), 127, dtype=np.uint8)
    y, _ = O.bmm_a8w8_ref(a, sa, w, sw)
    assert np.allclose(y[:, :, 0], A.sum(axis=-1), rtol=0, atol=1e-12 * np.abs(A).sum(axis=-1).max())
    assert np.array_equal(y[:, :, 1:], A)


def test_gemm_k_tail_equals_zero_padded():
    rng = np.random.Generator(np.random.PCG64(23))
    T, G, N = 2, 1, 5
    a = _rand_codes(rng, (T, G, 288))
    w = _rand_codes(rng, (G, N, 288))
    sa = rng.integers(118, 136, size=(T, G, 3), dtype=np.uint8)
    sw = rng.integers(118, 136, size=(G, N, 3), dtype=np.uint8)
    y, S = O.bmm_a8w8_ref(a, sa, w, sw)
    ap = np.zeros((T, G, 384), dtype=np.uint8)
    ap[..., :288] = a
    wp = np.zeros((G, N, 384), dtype=np.uint8)
    wp[..., :288] = w
    y2, S2 = O.bmm_a8w8_ref(ap, sa, wp, sw)
    assert np.array_equal(y, y2) and np.array_equal(S, S2)


def test_linear_against_bf16_dequant_path():
    """Loose pin against the pages' own unaligned-K path (BF16 activations times
    the dequantised weight): the difference is bounded by the activation
    quantisation error propagated through |W|."""
    M, N, K = 4, 32, 576
    x = W.bf16_normal((M, K), seed=31)
    wf = W.f32_normal((1, N, K), seed=32, std=0.02).numpy()
    wc, wsc = O.group_quant_rows(wf)
    y, S, a_codes, a_scales = O.linear_ref(W.bf16_bits(x), wc[0], wsc[0])
    Wv = O.mx_values(wc[0], wsc[0])
    xf = O.bf16_bits_to_f32(W.bf16_bits(x)).astype(np.float64)
    y_bf16path = xf @ Wv.T
    e = np.repeat(a_scales.astype(np.int64) - 127, 128, axis=-1)[:, :K]
    err_x = np.maximum(np.abs(xf) * 2.0 ** -4, np.ldexp(1.0, e - 10))
    bound = err_x @ np.abs(Wv).T + 1e-9
    assert np.all(np.abs(y - y_bf16path) <= bound)


def test_linear_handworked():
    """Hand-worked MXFP8 linear (tests/golden/linear_handworked.txt): the
    activation is quantised before the product (a tie rounded to the even
    code, a value rounded up to the next code, a partial 32-wide last group
    with its own scale), so y differs from the BF16 x times W product."""
    sec = read_sections("linear_handworked.txt")
    M, K, N = 2, 160, 3
    x = torch.zeros((M, K), dtype=torch.float32)
    for r, k, v in sec["x"]:
        x[int(r), int(k)] = float(v)
    x_bits = W.bf16_bits(x.to(torch.bfloat16))
    w = np.zeros((N, K), dtype=np.uint8)
    w[0, :] = 0x38
    w[1, 1] = 0x38
    w[2, 132] = 0x38
    sw = np.array([[127, 127], [127, 127], [127, 130]], dtype=np.uint8)
    y, S, a_codes, a_scales = O.linear_ref(x_bits, w, sw)
    want_codes = np.zeros((M, K), dtype=np.uint8)
    for r, k, c in sec["a_codes"]:
        want_codes[int(r), int(k)] = int(c, 16)
    want_scales = np.array([[int(b) for b in row[1:]] for row in sec["a_scales"]], dtype=np.uint8)
    want_y = np.zeros((M, N))
    want_S = np.zeros((M, N))
    for r, n, v in sec["y"]:
        want_y[int(r), int(n)] = float(v)
    for r, n, v in sec["S"]:
        want_S[int(r), int(n)] = float(v)
    assert np.array_equal(a_codes, want_codes)
    assert np.array_equal(a_scales, want_scales)
    assert np.array_equal(y, want_y)
    assert np.array_equal(S, want_S)


def test_gemm_tolerance_definition():
    y_ref = np.array([1.0, -3.0, 0.0])
    S = np.array([10.0, 0.0, 1.0])
    tol = O.gemm_tolerance(y_ref, S)
    assert np.allclose(tol, [2.0 ** -7 + 1e-4, 2.0 ** -6, 2.0 ** -133 + 1e-5], rtol=0, atol=0)
