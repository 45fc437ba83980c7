"""GPU parity of mxq_inv_rope_group_quant against the oracle: codes and
scale bytes must be bit-exact."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import oracle_quant, to_dev, wo_a_inputs
from conftest import read_sections
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    return m


def run(mxq, x, pos, cos, sin, R, err=None):
    xd, pd, cd, sd = to_dev(x, pos, cos, sin)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, R, err_flag=err)
    torch.cuda.synchronize()
    return q.cpu().numpy(), sc.cpu().numpy()


def assert_same(q, sc, q_ref, sc_ref):
    assert np.array_equal(sc, sc_ref), f"{np.sum(sc != sc_ref)} scale bytes differ"
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:4].tolist()}"


def test_tiny_config(mxq):
    # T=16, G=2, D=256, R=64, positions 0..15, seed 0
    x, pos, cos, sin = wo_a_inputs(16, 2, 256, 128, 64, seed=0, pos_mode="arange")
    q, sc = run(mxq, x, pos, cos, sin, 64)
    assert_same(q, sc, *oracle_quant(x, pos, cos, sin, 64))


def test_two_token_handworked(mxq):
    sec = read_sections("wo_a_2token_handworked.txt")
    x = torch.zeros((2, 1, 128), dtype=torch.float32)
    for t, k, v in sec["x"]:
        x[int(t), 0, int(k)] = float(v)
    x = x.to(torch.bfloat16)
    pos = torch.tensor([0, 1], dtype=torch.int64)
    cos, sin = W.rope_cache(2, 64)
    q, sc = run(mxq, x, pos, cos, sin, 64)
    codes = np.zeros((2, 1, 128), dtype=np.uint8)
    for t, k, c in sec["codes"]:
        codes[int(t), 0, int(k)] = int(c, 16)
    assert [int(b) for _, b in sec["scales"]] == list(sc[:, 0, 0])
    assert np.array_equal(q, codes)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_shapes(mxq, T):
    x, pos, cos, sin = wo_a_inputs(T, 8, 4096, 1024, 64, seed=300 + T, max_pos_table=32768)
    q, sc = run(mxq, x, pos, cos, sin, 64)
    assert_same(q, sc, *oracle_quant(x, pos, cos, sin, 64))


def test_prefill_chunk_sampled(mxq):
    """T=8192 (one 8K prefill chunk, 1% outliers x50), checked on 96 sampled
    tokens; plus a property over every group: its largest code magnitude lies
    in [224, 448] or its scale byte is 0."""
    T = 8192
    x, pos, cos, sin = wo_a_inputs(T, 8, 4096, 1024, 64, seed=400, pos_mode="arange",
                                   outlier_frac=0.01)
    xd, pd, cd, sd = to_dev(x, pos, cos, sin)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, 64)
    rng = np.random.Generator(np.random.PCG64(401))
    idx = np.unique(np.concatenate([[0, 1, T - 1], rng.integers(0, T, 93)]))
    q_ref, sc_ref = oracle_quant(x[idx], pos[idx], cos, sin, 64)
    assert_same(q[idx].cpu().numpy(), sc[idx].cpu().numpy(), q_ref, sc_ref)
    lut = torch.from_numpy(np.abs(np.nan_to_num(O.E4M3_TABLE)).astype(np.float32)).to(q.device)
    mags = lut[q.long()].view(T, 8, 32, 128).amax(dim=-1)
    okay = ((mags >= 224) & (mags <= 448)) | (sc == 0)
    assert bool(okay.all())


@pytest.mark.parametrize("D", [16, 144, 288, 576, 2304])
def test_partial_last_group_no_rope(mxq, D):
    x = W.bf16_normal((7, 3, D), seed=D)
    pos = torch.zeros(7, dtype=torch.int64)
    cos, sin = W.rope_cache(1, 2)
    q, sc = run(mxq, x, pos, cos, sin, 0)
    assert_same(q, sc, *oracle_quant(x, pos, cos, sin, 0))


@pytest.mark.parametrize("R", [16, 32, 48, 128])
def test_rope_widths(mxq, R):
    x, pos, cos, sin = wo_a_inputs(9, 2, 384, 128, R, seed=500 + R, max_pos=4096)
    q, sc = run(mxq, x, pos, cos, sin, R)
    assert_same(q, sc, *oracle_quant(x, pos, cos, sin, R))


def test_strided_cos_sin_view(mxq):
    """cos/sin rows taken from a wider cache (leading dimension 48 > R/2)."""
    x, pos, _, _ = wo_a_inputs(12, 2, 256, 128, 64, seed=600, max_pos=1000)
    cos_w, sin_w = W.rope_cache(1000, 96)  # [1000, 48]
    cos, sin = cos_w[:, :32], sin_w[:, :32]
    xd, pd, cd, sd = to_dev(x, pos, cos_w, sin_w)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd[:, :32], sd[:, :32], 64)
    torch.cuda.synchronize()
    assert cd[:, :32].stride(0) == 48
    # The oracle indexes entries 0..R/2-1 of each row of the same numbers.
    assert_same(q.cpu().numpy(), sc.cpu().numpy(),
                *oracle_quant(x, pos, cos.contiguous(), sin.contiguous(), 64))


def test_special_values(mxq):
    """Zero groups (scale byte 0), negative zeros, BF16 subnormals, huge
    finite values, and values that round across E4M3 binades."""
    T, G, D = 4, 1, 512
    v = np.zeros((T, G, D), dtype=np.float32)
    v[0, 0, 128:256] = -0.0
    v[1, 0, :128] = 1e-39  # BF16/FP32 subnormal amax -> scale byte 0
    v[1, 0, 5] = -3e-39
    v[2, 0, :128] = np.linspace(-3e38, 3e38, 128, dtype=np.float32)
    v[2, 0, 128:256] = np.float32(15.5) * np.arange(-64, 64, dtype=np.float32)
    v[3, 0, :] = np.float32(2.0) ** np.arange(-64, 64, 0.25, dtype=np.float32)[:512]
    x = torch.from_numpy(v).to(torch.bfloat16)
    pos = torch.arange(T, dtype=torch.int64)
    cos, sin = W.rope_cache(T, 64)
    q, sc = run(mxq, x, pos, cos, sin, 64)
    assert_same(q, sc, *oracle_quant(x, pos, cos, sin, 64))
    assert sc[0, 0, 0] == 0 and sc[0, 0, 1] == 0
    assert (q[0, 0, 128:256] == 0x80).all()


def test_out_of_range_position_sets_flag_and_zeroes_row(mxq):
    T = 6
    x, _, cos, sin = wo_a_inputs(T, 2, 256, 128, 64, seed=700, max_pos=100, max_pos_table=100)
    pos = torch.tensor([3, -1, 50, 100, 99, 7], dtype=torch.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, sc = run(mxq, x, pos, cos, sin, 64, err=err)
    assert int(err.item()) == mxq.MXQ_DEVERR_POSITION
    for t in (1, 3):
        assert (q[t] == 0).all() and (sc[t] == 0).all()
    good = np.array([0, 2, 4, 5])
    q_ref, sc_ref = oracle_quant(x[good], pos[good], cos, sin, 64)
    assert_same(q[good], sc[good], q_ref, sc_ref)


def test_valid_positions_leave_flag_clear(mxq):
    x, pos, cos, sin = wo_a_inputs(5, 2, 256, 128, 64, seed=710, max_pos=50)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    run(mxq, x, pos, cos, sin, 64, err=err)
    assert int(err.item()) == 0


def test_empty_input_is_noop(mxq):
    x = torch.empty((0, 8, 4096), dtype=torch.bfloat16, device="cuda")
    pos = torch.empty((0,), dtype=torch.int64, device="cuda")
    cos, sin = to_dev(*W.rope_cache(4, 64))
    q, sc = mxq.mxq_inv_rope_group_quant(x, pos, cos, sin, 64)
    assert q.shape == (0, 8, 4096) and sc.shape == (0, 8, 32)


def test_maximum_row_length(mxq):
    """D = 65536 (512 scale groups per row, the largest D the ABI accepts) with
    the widest rotated slice, R = 128."""
    x, pos, cos, sin = wo_a_inputs(40, 2, 65536, 16, 128, seed=2200, max_pos=5000)
    q, sc = run(mxq, x, pos, cos, sin, 128)
    assert_same(q, sc, *oracle_quant(x, pos, cos, sin, 128))
