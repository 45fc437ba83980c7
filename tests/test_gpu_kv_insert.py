"""GPU parity of mxq_rope_kv_insert (forward RoPE of the query and of the new
KV row, KV row stored in an OCP E4M3 cache with a per-tensor scale or in a
BF16 cache) against the oracle, bit for bit: the query bits, every cache
byte (rows not addressed must keep their previous contents) and the device
error word."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import to_dev
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    return m


def inputs(T, H, Dq, Dk, R, seed, max_pos=32768, num_slots=None, kv_std=4.0):
    q = W.bf16_normal((T, H, Dq), seed=seed)
    kv = W.bf16_normal((T, Dk), seed=seed + 1, std=kv_std)
    pos = W.positions_uniform(T, seed=seed + 2, max_pos=max_pos)
    cos, sin = W.rope_cache(max_pos, max(R, 2))
    num_slots = num_slots or 2 * T + 3
    rng = np.random.Generator(np.random.PCG64(seed + 3))
    slots = rng.permutation(num_slots)[:T].astype(np.int64)
    return q, kv, pos, cos, sin, slots, num_slots


def run(mxq, q, kv, pos, cos, sin, R, slots, num_slots, scale, inplace=False, fill=0xA5):
    T, Dk = kv.shape
    qd, kvd, pd, cd, sd = to_dev(q, kv, pos, cos, sin)
    sl = torch.from_numpy(slots).cuda()
    if scale is None:
        v = fill * 257
        cache = torch.full((num_slots, Dk), v - 65536 if v >= 32768 else v, dtype=torch.int16,
                           device="cuda").view(torch.bfloat16)
        sc = None
    else:
        cache = torch.full((num_slots, Dk), fill, dtype=torch.uint8, device="cuda")
        sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_out = mxq.mxq_rope_kv_insert(qd, kvd, pd, cd, sd, R, sl, cache, scale=sc,
                                   q_out=qd if inplace else None, err_flag=err)
    torch.cuda.synchronize()
    return q_out, cache, int(err.item()), qd


def oracle(q, kv, pos, cos, sin, R, slots, num_slots, scale, fill=0xA5):
    Dk = kv.shape[1]
    if scale is None:
        cache = np.full((num_slots, Dk), fill * 257, dtype=np.uint16)
    else:
        cache = np.full((num_slots, Dk), fill, dtype=np.uint8)
    return O.rope_kv_insert(W.bf16_bits(q), W.bf16_bits(kv), pos.numpy(), W.bf16_bits(cos),
                            W.bf16_bits(sin), R, slots, cache, scale=scale)


def cache_bits(cache):
    if cache.dtype == torch.bfloat16:
        return W.bf16_bits(cache.cpu())
    return cache.cpu().numpy()


@pytest.mark.parametrize("scale", [0.0371, 0.5, None])
@pytest.mark.parametrize("T", [1, 8, 64])
def test_decode_shapes(mxq, T, scale):
    """q [T, 64, 512], kv [T, 512], R = 64 at random positions below 32768;
    E4M3 cache with a non-power-of-two and a power-of-two scale, and BF16."""
    q, kv, pos, cos, sin, slots, ns = inputs(T, 64, 512, 512, 64, seed=5000 + T, num_slots=4096)
    q_out, cache, err, _ = run(mxq, q, kv, pos, cos, sin, 64, slots, ns, scale)
    want_q, want_cache = oracle(q, kv, pos, cos, sin, 64, slots, ns, scale)
    assert err == 0
    assert np.array_equal(W.bf16_bits(q_out.cpu()), want_q)
    assert np.array_equal(cache_bits(cache), want_cache)


@pytest.mark.parametrize("R", [0, 16, 32, 128])
@pytest.mark.parametrize("scale", [0.0371, None])
def test_ragged_shapes_and_widths(mxq, R, scale):
    """T = 37 tokens, 3 heads of 192, KV rows of 576 (the rotated slice ends
    the row, R from none to 128)."""
    q, kv, pos, cos, sin, slots, ns = inputs(37, 3, 192, 576, R, seed=5100 + R, max_pos=5000)
    q_out, cache, err, _ = run(mxq, q, kv, pos, cos, sin, R, slots, ns, scale)
    want_q, want_cache = oracle(q, kv, pos, cos, sin, R, slots, ns, scale)
    assert err == 0
    assert np.array_equal(W.bf16_bits(q_out.cpu()), want_q)
    assert np.array_equal(cache_bits(cache), want_cache)


@pytest.mark.parametrize("scale", [0.0371, None])
def test_query_in_place(mxq, scale):
    q, kv, pos, cos, sin, slots, ns = inputs(20, 8, 512, 512, 64, seed=5200)
    q_out, cache, err, qd = run(mxq, q, kv, pos, cos, sin, 64, slots, ns, scale, inplace=True)
    want_q, want_cache = oracle(q, kv, pos, cos, sin, 64, slots, ns, scale)
    assert q_out.data_ptr() == qd.data_ptr() and err == 0
    assert np.array_equal(W.bf16_bits(q_out.cpu()), want_q)
    assert np.array_equal(cache_bits(cache), want_cache)


def test_no_query_and_padding_slots(mxq):
    """H = 0 (KV rows only); negative slots (padding tokens) write nothing."""
    T, Dk = 50, 256
    _, kv, pos, cos, sin, slots, ns = inputs(T, 1, 16, Dk, 64, seed=5300)
    slots[::3] = -1
    kvd, pd, cd, sd = to_dev(kv, pos, cos, sin)
    cache = torch.full((ns, Dk), 0x77, dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.25], dtype=torch.float32, device="cuda")
    st = mxq.lib().mxq_rope_kv_insert(None, None, T, 0, 0, mxq._ptr(kvd), Dk, mxq._ptr(pd),
                                      mxq._ptr(cd), mxq._ptr(sd), cd.stride(0), cd.shape[0], 64,
                                      mxq._ptr(torch.from_numpy(slots).cuda()), mxq._ptr(cache), ns,
                                      mxq.MXQ_CACHE_E4M3, mxq._ptr(sc), None, mxq._stream(None))
    assert st == 0, mxq.lib().mxq_last_error()
    torch.cuda.synchronize()
    q0 = torch.zeros((T, 1, 64), dtype=torch.bfloat16)
    _, want = O.rope_kv_insert(W.bf16_bits(q0), W.bf16_bits(kv), pos.numpy(), W.bf16_bits(cos),
                               W.bf16_bits(sin), 64, slots, np.full((ns, Dk), 0x77, dtype=np.uint8),
                               scale=0.25)
    assert np.array_equal(cache.cpu().numpy(), want)


def test_invalid_positions_and_slots(mxq):
    """A position outside the table: that token's query slices are zero, its
    KV row is not written, MXQ_DEVERR_POSITION; a slot >= num_slots: no row,
    MXQ_DEVERR_SLOT.  Every other token as the oracle."""
    T, H, D, R = 12, 4, 256, 64
    q, kv, pos, cos, sin, slots, ns = inputs(T, H, D, D, R, seed=5400, max_pos=100)
    pos[[2, 7]] = torch.tensor([100, -3], dtype=torch.int64)
    slots[5] = ns
    q_out, cache, err, _ = run(mxq, q, kv, pos, cos, sin, R, slots, ns, 0.125)
    assert err == mxq.MXQ_DEVERR_POSITION | mxq.MXQ_DEVERR_SLOT
    good = np.array([t for t in range(T) if t not in (2, 7)])
    g_slots = slots[good].copy()
    g_slots[g_slots >= ns] = -1
    want_q, want_cache = oracle(q[good], kv[good], pos[good], cos, sin, R, g_slots, ns, 0.125)
    got_q = W.bf16_bits(q_out.cpu())
    assert np.array_equal(got_q[good], want_q)
    qb = W.bf16_bits(q)
    for t in (2, 7):
        assert (got_q[t, :, D - R:] == 0).all()
        assert np.array_equal(got_q[t, :, :D - R], qb[t, :, :D - R])
    assert np.array_equal(cache.cpu().numpy(), want_cache)


def test_prefill_chunk(mxq):
    """8192 tokens at positions 32768..40959, q [8192, 64, 512], kv [8192, 512]
    into an E4M3 cache of 16384 rows: every cache byte against the oracle,
    the query on sampled tokens."""
    T, H, D, R = 8192, 64, 512, 64
    q = W.bf16_normal((T, H, D), seed=5500)
    kv = W.bf16_normal((T, D), seed=5501, std=4.0)
    pos = W.positions_arange(32768, T)
    cos, sin = W.rope_cache(40960, R)
    ns = 16384
    slots = np.random.Generator(np.random.PCG64(5502)).permutation(ns)[:T].astype(np.int64)
    q_out, cache, err, _ = run(mxq, q, kv, pos, cos, sin, R, slots, ns, 0.0371)
    assert err == 0
    kv_q0 = torch.zeros((T, 1, 64), dtype=torch.bfloat16)
    _, want_cache = O.rope_kv_insert(W.bf16_bits(kv_q0), W.bf16_bits(kv), pos.numpy(),
                                     W.bf16_bits(cos), W.bf16_bits(sin), R, slots,
                                     np.full((ns, D), 0xA5, dtype=np.uint8), scale=0.0371)
    assert np.array_equal(cache.cpu().numpy(), want_cache)
    idx = np.unique(np.concatenate([[0, 1, 4095, 4096, T - 1],
                                    np.random.Generator(np.random.PCG64(5503)).integers(0, T, 27)]))
    want_q, _ = O.rope_kv_insert(W.bf16_bits(q[idx]), W.bf16_bits(kv[idx]), pos[idx].numpy(),
                                 W.bf16_bits(cos), W.bf16_bits(sin), R, -np.ones(len(idx), np.int64),
                                 np.zeros((1, D), dtype=np.uint8), scale=0.0371)
    assert np.array_equal(W.bf16_bits(q_out[idx].cpu()), want_q)


def test_strided_cos_sin_views(mxq):
    """cos/sin as column slices of a wider cache (row stride 48 > R/2 = 32):
    only the first R/2 entries of each row are used."""
    T, H, D, R = 16, 4, 256, 64
    q, kv, pos, _, _, slots, ns = inputs(T, H, D, D, R, seed=5600, max_pos=300)
    cw, swide = W.rope_cache(300, 96)  # 48 entries per row
    cos, sin = cw[:, :32], swide[:, :32]
    qd, kvd, pd = to_dev(q, kv, pos)
    cdw, sdw = to_dev(cw, swide)
    cache = torch.full((ns, D), 0xA5, dtype=torch.uint8, device="cuda")
    sc = torch.tensor([0.0371], dtype=torch.float32, device="cuda")
    q_out = mxq.mxq_rope_kv_insert(qd, kvd, pd, cdw[:, :32], sdw[:, :32], R,
                                   torch.from_numpy(slots).cuda(), cache, scale=sc)
    torch.cuda.synchronize()
    want_q, want_cache = O.rope_kv_insert(W.bf16_bits(q), W.bf16_bits(kv), pos.numpy(),
                                          W.bf16_bits(cos.contiguous()), W.bf16_bits(sin.contiguous()), R,
                                          slots, np.full((ns, D), 0xA5, dtype=np.uint8), scale=0.0371)
    assert np.array_equal(W.bf16_bits(q_out.cpu()), want_q)
    assert np.array_equal(cache.cpu().numpy(), want_cache)


@pytest.mark.parametrize("R,scale", [(64, 0.0371), (0, None), (128, 0.5)])
def test_streaming_query_path(mxq, R, scale):
    """Out-of-place queries of 32 MiB or more go through the streaming kernel
    (blocks of whole rows rotated in shared memory): T = 2000 tokens of 16
    heads x 576 (28 rows per 32 KB block, so blocks straddle tokens and the
    last block is short), two tokens at invalid positions (their query slices
    zero, their KV rows not written, MXQ_DEVERR_POSITION), every query bit
    and cache byte against the oracle."""
    T, H, D, Dk = 2000, 16, 576, 576
    assert T * H * D * 2 >= 32 << 20 and (T * H) % 28 != 0
    q, kv, pos, cos, sin, slots, ns = inputs(T, H, D, Dk, max(R, 16), seed=5700 + R, max_pos=4000)
    bad = [] if R == 0 else [45, 1711]
    if bad:
        pos[bad] = torch.tensor([4000, -2], dtype=torch.int64)
    q_out, cache, err, _ = run(mxq, q, kv, pos, cos, sin, R, slots, ns, scale)
    assert err == (mxq.MXQ_DEVERR_POSITION if bad else 0)
    good = np.array([t for t in range(T) if t not in bad])
    g_slots = slots.copy()
    g_slots[bad] = -1
    want_q, want_cache = oracle(q[good], kv[good], pos[good], cos, sin, R, g_slots[good], ns, scale)
    got_q = W.bf16_bits(q_out.cpu())
    assert np.array_equal(got_q[good], want_q)
    qb = W.bf16_bits(q)
    for t in bad:
        assert (got_q[t, :, D - R:] == 0).all()
        assert np.array_equal(got_q[t, :, :D - R], qb[t, :, :D - R])
    assert np.array_equal(cache_bits(cache), want_cache)
