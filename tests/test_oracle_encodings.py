"""Pins of the oracle's number formats against things other than itself:
hand-worked values, torch's own float8_e4m3fn / bfloat16 conversions, and
the brute-force definition of the scale rule."""

import math

import numpy as np
import pytest
import torch

from conftest import parse_float, read_table
from oracle import mx_oracle as O


def test_e4m3_table_textbook_values():
    t = O.E4M3_TABLE
    assert t[0x38] == 1.0
    assert t[0x7E] == 448.0
    assert t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9
    assert t[0x07] == 7 * 2.0 ** -9
    assert t[0x08] == 2.0 ** -6
    assert t[0x40] == 2.0
    assert t[0x00] == 0.0 and not math.copysign(1.0, t[0x00]) < 0
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) < 0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert np.sum(np.isnan(t)) == 2


def test_e4m3_table_matches_torch_decode():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    both_nan = np.isnan(ref) & np.isnan(O.E4M3_TABLE)
    assert np.all(both_nan | (ref == O.E4M3_TABLE))
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(O.E4M3_TABLE[~both_nan]))


@pytest.mark.parametrize("row", read_table("e4m3_encode_handworked.txt"), ids=lambda r: r[0])
def test_e4m3_encode_handworked(row):
    v, code = parse_float(row[0]), int(row[1], 16)
    assert int(O.e4m3_encode(np.array([v]))[0]) == code


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_on_midpoints():
    pos = O.E4M3_TABLE[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2.0  # exact in fp32 (few significant bits)
    m32 = mids.astype(np.float32)
    cand = np.concatenate([m32, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9)),
                           pos.astype(np.float32)])
    cand = cand[np.abs(cand) <= 448.0]
    cand = np.concatenate([cand, -cand])
    ours = O.e4m3_encode(cand.astype(np.float64))
    assert np.array_equal(ours, _torch_e4m3(cand))


def test_e4m3_encode_matches_torch_random():
    rng = np.random.Generator(np.random.PCG64(7))
    # log-uniform magnitudes across the whole E4M3 range incl. subnormals and underflow
    mag = np.exp2(rng.uniform(-14.0, math.log2(448.0), size=400_000)).astype(np.float32)
    sign = np.where(rng.random(400_000) < 0.5, -1.0, 1.0).astype(np.float32)
    v = mag * sign
    v = v[np.abs(v) <= 448.0]
    assert np.array_equal(O.e4m3_encode(v.astype(np.float64)), _torch_e4m3(v))


def test_e4m3_encode_saturates():
    v = np.array([448.0, 448.5, 460.0, 1e6, 3e38, -449.0, -1e30])
    assert list(O.e4m3_encode(v)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_e4m3_encode_nan_gives_a_nan_code():
    """NaN has a code of its own in e4m3fn (S.1111.111); encoding keeps it NaN
    rather than saturating it to +-448."""
    codes = O.e4m3_encode(np.array([np.nan, -np.nan, np.nan * 0.0]))
    assert all(int(c) & 0x7F == 0x7F for c in codes)
    assert np.isnan(O.e4m3_decode(codes)).all()


@pytest.mark.parametrize("row", read_table("e8m0_scale_handworked.txt"), ids=lambda r: r[0])
def test_scale_rule_handworked(row):
    amax, byte = parse_float(row[0]), int(row[1])
    amax = float(np.float32(amax))  # amax is an fp32 magnitude in the kernel
    assert int(O.e8m0_exponent(np.array([amax]))[0]) + 127 == byte


def _scale_by_definition(amax):
    """Smallest e in [-127, 127] with amax <= 448 * 2^e (plain loop)."""
    for e in range(-127, 128):
        if amax <= math.ldexp(448.0, e):
            return e
    return 127


def test_scale_rule_brute_force():
    rng = np.random.Generator(np.random.PCG64(11))
    bits = rng.integers(0, 0x7F800000, size=20_000, dtype=np.uint32)  # all finite fp32 >= 0
    amax = bits.view(np.float32).astype(np.float64)
    # beyond fp32 too: the clamp at 127 is part of the rule's definition
    amax = np.concatenate([amax, [0.0, 448.0, 448.00003, 1.0, 2.0 ** -149, 3.4e38, 2.0 ** 200, 1e300]])
    e = O.e8m0_exponent(amax)
    for a, ee in zip(amax, e):
        assert ee == _scale_by_definition(a), a


def test_scale_rule_invariant():
    rng = np.random.Generator(np.random.PCG64(12))
    amax = np.exp2(rng.uniform(-110, 120, size=100_000))
    e = O.e8m0_exponent(amax)
    r = np.ldexp(amax, -e)
    assert np.all((r > 224.0) & (r <= 448.0))


@pytest.mark.parametrize("row", read_table("dequant_handworked.txt"), ids=lambda r: r[0] + "_" + r[1])
def test_dequant_handworked(row):
    code, sc = int(row[0], 16), int(row[1])
    got = int(O.dequant_bf16(np.array([[code]], dtype=np.uint8), np.array([[sc]], dtype=np.uint8))[0, 0])
    if row[2] == "NAN":
        assert (got & 0x7F80) == 0x7F80 and (got & 0x7F) != 0
    else:
        assert got == int(row[2], 16), hex(got)


def test_dequant_exhaustive_matches_torch():
    """Every (code, scale byte) pair against torch: the exact product (fits in
    float32, or overflows it exactly when it also overflows BF16), then torch's
    float32 -> bfloat16 round-to-nearest-even."""
    codes = np.repeat(np.arange(256, dtype=np.uint8), 256)
    scs = np.tile(np.arange(256, dtype=np.uint8), 256)
    ours = O.dequant_bf16(codes[:, None], scs[:, None])[:, 0]
    dec = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    val = dec[torch.from_numpy(codes.astype(np.int64))] * torch.pow(
        torch.tensor(2.0, dtype=torch.float64), torch.from_numpy(scs.astype(np.float64)) - 127.0)
    val[torch.from_numpy(scs == 255)] = float("nan")
    ref = val.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan_ref = (ref & 0x7F80) == 0x7F80
    nan_ref &= (ref & 0x7F) != 0
    nan_ours = ((ours & 0x7F80) == 0x7F80) & ((ours & 0x7F) != 0)
    assert np.array_equal(nan_ref, nan_ours)
    assert np.array_equal(ours[~nan_ref], ref[~nan_ref])


def test_bf16_rne_matches_torch():
    rng = np.random.Generator(np.random.PCG64(13))
    bits = rng.integers(0, 0xFFFFFFFF, size=300_000, dtype=np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    ours = O.bf16_rne_bits(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_ulp():
    u = O.bf16_ulp(np.array([1.0, 1.5, -3.0, 2.0 ** -130, 0.0, 2.0 ** -126, 255.0]))
    assert list(u) == [2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -133, 2.0 ** -133, 2.0 ** -133, 1.0]


def test_scales_f32_to_e8m0():
    ks = np.arange(-127, 128)
    s = np.ldexp(np.ones(ks.shape), ks).astype(np.float32)
    out, ok = O.scales_f32_to_e8m0(s)
    assert ok.all() and np.array_equal(out, (ks + 127).astype(np.uint8))
    bad = np.array([0.0, -1.0, 3.0, 0.75, np.inf, np.nan, 2.0 ** -128, 2.0 ** -149, -0.5], dtype=np.float32)
    out, ok = O.scales_f32_to_e8m0(bad)
    assert not ok.any() and (out == 0xFF).all()
