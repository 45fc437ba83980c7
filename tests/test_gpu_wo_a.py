"""GPU parity of mxq_wo_a, the whole wo_a projection in one call (one fused
launch for T <= 32, quantiser + GEMM through a workspace for 32 < T <= 128,
one launch of the quantising CTA-pair GEMM above), against the oracle:
inverse RoPE + group quantisation, then the block-scaled GEMM."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import check_gemm, oracle_quant, oracle_weights, to_dev, wo_a_inputs
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    m.mxq_watchdog_read(clear=True)
    yield m
    assert m.mxq_watchdog_read() == 0


def run(mxq, x, pos, cos, sin, w, sw, R, err=None):
    D = x.shape[-1]
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, D)
    out = mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=R, err_flag=err)
    torch.cuda.synchronize()
    return out, (xd, pd, cd, sd, wd, wsf)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_shapes_one_launch(mxq, T):
    """x [T, 8, 4096] at random positions in [0, 32768), W [8, 1024, 4096]."""
    x, pos, cos, sin = wo_a_inputs(T, 8, 4096, 1024, 64, seed=1300 + T, max_pos_table=32768)
    w, sw = oracle_weights(8, 1024, 4096, seed=3)
    out, _ = run(mxq, x, pos, cos, sin, w, sw, 64)
    a, sa = oracle_quant(x, pos, cos, sin, 64)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"wo_a T={T}")


@pytest.mark.parametrize("R", [0, 16, 32, 64, 128])
@pytest.mark.parametrize("T", [3, 17, 33, 63])
def test_ragged_tokens_and_rope_widths(mxq, T, R):
    x, pos, cos, sin = wo_a_inputs(T, 2, 512, 256, max(R, 16), seed=1400 + T + R, max_pos=5000)
    w, sw = oracle_weights(2, 256, 512, seed=1401)
    out, _ = run(mxq, x, pos, cos, sin, w, sw, R)
    a, sa = oracle_quant(x, pos, cos, sin, R)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"T={T} R={R}")


@pytest.mark.parametrize("T", [33, 65, 100, 128, 129, 300])
def test_larger_token_counts(mxq, T):
    """Both sides of each boundary between the forms (32/33, 128/129)."""
    x, pos, cos, sin = wo_a_inputs(T, 2, 1024, 256, 64, seed=1500 + T, max_pos=4096)
    w, sw = oracle_weights(2, 256, 1024, seed=1501)
    out, _ = run(mxq, x, pos, cos, sin, w, sw, 64)
    a, sa = oracle_quant(x, pos, cos, sin, 64)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"T={T}")


@pytest.mark.parametrize("D", [288, 576, 2304])
def test_unaligned_k_without_rope(mxq, D):
    x, pos, cos, sin = wo_a_inputs(8, 2, D, 512, 16, seed=1600 + D, max_pos=64)
    w, sw = oracle_weights(2, 512, D, seed=1601 + D)
    out, _ = run(mxq, x, pos, cos, sin, w, sw, 0)
    a, sa = oracle_quant(x, pos, cos, sin, 0)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"D={D}")


@pytest.mark.parametrize("T", [1, 8, 32])
def test_one_launch_matches_two_calls(mxq, T):
    """The fused launch and the quantiser + GEMM sequence agree within the GEMM
    tolerance (the two may split K differently, so fp32 sums can differ in the
    last place; the quantised operands are the same)."""
    x, pos, cos, sin = wo_a_inputs(T, 8, 4096, 1024, 64, seed=1700 + T, max_pos_table=32768)
    w, sw = oracle_weights(8, 1024, 4096, seed=3)
    out, (xd, pd, cd, sd, wd, wsf) = run(mxq, x, pos, cos, sin, w, sw, 64)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, 64)
    out2 = mxq.mxq_bmm_a8w8(q, sc, wd, wsf)
    torch.cuda.synchronize()
    a, sa = oracle_quant(x, pos, cos, sin, 64)
    y_ref, S = O.bmm_a8w8_ref(a, sa, w, sw)
    assert np.array_equal(q.cpu().numpy(), a) and np.array_equal(sc.cpu().numpy(), sa)
    y1 = out.float().cpu().numpy().astype(np.float64)
    y2 = out2.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y1 - y2) <= O.gemm_tolerance(y2, S))
    check_gemm(out, y_ref, S, "fused")


def test_out_of_range_position_in_one_launch(mxq):
    T = 6
    x, _, cos, sin = wo_a_inputs(T, 2, 256, 128, 64, seed=1800, max_pos=100, max_pos_table=100)
    pos = torch.tensor([3, -1, 50, 100, 99, 7], dtype=torch.int64)
    w, sw = oracle_weights(2, 128, 256, seed=1801)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = run(mxq, x, pos, cos, sin, w, sw, 64, err=err)
    assert int(err.item()) == mxq.MXQ_DEVERR_POSITION
    o = out.float().cpu()
    assert (o[1] == 0).all() and (o[3] == 0).all()
    good = np.array([0, 2, 4, 5])
    a, sa = oracle_quant(x[good], pos[good], cos, sin, 64)
    check_gemm(out[good], *O.bmm_a8w8_ref(a, sa, w, sw), "good rows")


# ----------------------------------------------------------------------------
# Above 128 tokens mxq_wo_a is one launch of the CTA-pair GEMM whose extra
# warps quantise the activation into the workspace: codes [T, G, D], scale
# atoms [G, MB, KG, 512] (MB = 2 * ceil(T / 256) blocks of 128 tokens; row r of
# a block holds its scale byte four times at (r % 32) * 16 + (r // 32) * 4) and
# one uint32 job counter per (g, block, k group), raised once for each of the
# 8 slices of 16 rows that the CTA owning the block quantises.

def ws_layout(T, G, D):
    r256 = lambda v: (v + 255) // 256 * 256
    MB = 2 * ((T + 255) // 256)
    KG = (D + 127) // 128
    jobs = G * MB * KG
    atoms = r256(T * G * D)
    flags = atoms + r256(jobs * 512)
    return atoms, flags, flags + r256(jobs * 4), MB, KG


def atom_scales(ws, T, G, D):
    """Scale bytes [T, G, KG] read back from the workspace's atoms (each word must
    hold one byte four times; rows past T must hold 127)."""
    atoms, flags, _, MB, KG = ws_layout(T, G, D)
    at = ws[atoms:atoms + G * MB * KG * 512].cpu().numpy().reshape(G, MB, KG, 32, 4, 4)
    assert (at == at[..., :1]).all(), "an atom word does not repeat its byte"
    # [G, MB, KG, line r%32, word r//32] -> [G, MB, r, KG]
    b = at[..., 0].transpose(0, 1, 4, 3, 2).reshape(G, MB * 128, KG)
    assert (b[:, T:, :] == 127).all()
    return b[:, :T, :].transpose(1, 0, 2)


@pytest.mark.parametrize("T,G,D,N,R", [
    (129, 1, 256, 16, 64),      # one token in the second pair half
    (257, 2, 512, 272, 16),     # odd CTA of the second block almost empty
    (300, 3, 640, 1040, 128),   # five weight tiles, the last mostly past N
    (1000, 2, 1024, 256, 64),   # one weight tile: each pair quantises all K groups
    (384, 2, 576, 512, 0),      # unaligned K (4 groups + 64), no rotation
    (520, 1, 2304, 768, 0),     # unaligned K (18 groups), three weight tiles
])
def test_pair_quant_workspace_and_output(mxq, T, G, D, N, R):
    x, pos, cos, sin = wo_a_inputs(T, G, D, N, max(R, 16), seed=1900 + T + D, max_pos=5000)
    w, sw = oracle_weights(G, N, D, seed=1901 + D)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, D)
    atoms, flags, total, MB, KG = ws_layout(T, G, D)
    assert mxq.mxq_wo_a_workspace_bytes(T, G, D, N) == total
    ws = torch.full((total,), 0xA5, dtype=torch.uint8, device="cuda")
    out = mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=R, ws=ws)
    torch.cuda.synchronize()
    a, sa = oracle_quant(x, pos, cos, sin, R)
    codes = ws[:T * G * D].cpu().numpy().reshape(T, G, D)
    assert np.array_equal(codes, a), "codes differ from the oracle"
    assert np.array_equal(atom_scales(ws, T, G, D), sa), "scale bytes differ from the oracle"
    cnt = ws[flags:flags + G * MB * KG * 4].cpu().view(torch.int32).numpy()
    assert (cnt == 8).all(), "a job counter is not 8"
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"pair quant T={T} D={D} N={N} R={R}")
    # Same operands, same MMA sequence: bit-identical to quantiser + GEMM.
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, R)
    out2 = mxq.mxq_bmm_a8w8(q, sc, wd, wsf)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_pair_quant_out_of_range_positions(mxq):
    T, G, D, N = 300, 2, 512, 256
    x, _, cos, sin = wo_a_inputs(T, G, D, N, 64, seed=2000, max_pos=100, max_pos_table=100)
    rng = np.random.Generator(np.random.PCG64(2001))
    pos = torch.from_numpy(rng.integers(0, 100, T).astype(np.int64))
    bad = np.array([0, 5, 128, 200, 299])
    pos[bad] = torch.tensor([-1, 100, 1000, -7, 100], dtype=torch.int64)
    w, sw = oracle_weights(G, N, D, seed=2002)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = run(mxq, x, pos, cos, sin, w, sw, 64, err=err)
    assert int(err.item()) == mxq.MXQ_DEVERR_POSITION
    o = out.float().cpu()
    assert (o[bad] == 0).all()
    good = np.setdiff1d(np.arange(T), bad)
    a, sa = oracle_quant(x[good], pos[good], cos, sin, 64)
    check_gemm(out[good], *O.bmm_a8w8_ref(a, sa, w, sw), "good rows")


def test_pair_quant_deterministic_and_graph_replay(mxq):
    """Repeated calls, eager and replayed from a CUDA graph (the counters are
    cleared inside each call), give identical outputs."""
    T, G, D, N = 700, 4, 1024, 512
    x, pos, cos, sin = wo_a_inputs(T, G, D, N, 64, seed=2100, max_pos=4096)
    w, sw = oracle_weights(G, N, D, seed=2101)
    out, (xd, pd, cd, sd, wd, wsf) = run(mxq, x, pos, cos, sin, w, sw, 64)
    ws = torch.empty(mxq.mxq_wo_a_workspace_bytes(T, G, D, N), dtype=torch.uint8, device="cuda")
    o2 = torch.empty_like(out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=64, out=o2, ws=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(out, o2)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=64, out=o2, ws=ws,
                     stream=torch.cuda.current_stream())
    for _ in range(3):
        o2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o2)


def test_pair_quant_repeated_runs_match_two_kernels(mxq):
    """Production G, D, N at 2048 tokens, 20 calls on one workspace: every
    output bit-identical to quantiser + GEMM (a missing ordering between the
    quantising warps and the consuming CTAs would show as a sporadic
    mismatch), and the first also against the oracle on sampled tokens."""
    T, G, D, N = 2048, 8, 4096, 1024
    x, pos, cos, sin = wo_a_inputs(T, G, D, N, 64, seed=2200, pos_mode="arange",
                                   outlier_frac=0.01)
    w, sw = oracle_weights(G, N, D, seed=3)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, D)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, 64)
    ref = mxq.mxq_bmm_a8w8(q, sc, wd, wsf)
    ws = torch.empty(mxq.mxq_wo_a_workspace_bytes(T, G, D, N), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(ref)
    for i in range(20):
        mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=64, out=out, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {i} differs from quantiser + GEMM"
        if i == 0:
            idx = np.array([0, 127, 128, 1000, 2047])
            a, sa = oracle_quant(x[idx], pos[idx], cos, sin, 64)
            check_gemm(out[idx], *O.bmm_a8w8_ref(a, sa, w, sw), "sampled")


@pytest.mark.parametrize("T", [8, 64, 160])
def test_maximum_d(mxq, T):
    """D = K = 65536, the largest row the ABI accepts (512 scale groups, the
    rotated slice in the last one), through the fused decode launch (T = 8),
    quantiser + GEMM (T = 64) and the quantising CTA-pair launch (T = 160)."""
    x, pos, cos, sin = wo_a_inputs(T, 1, 65536, 16, 64, seed=2100 + T, max_pos=5000)
    w, sw = oracle_weights(1, 16, 65536, seed=2101)
    out, _ = run(mxq, x, pos, cos, sin, w, sw, 64)
    a, sa = oracle_quant(x, pos, cos, sin, 64)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"D=65536 T={T}")


@pytest.mark.parametrize("pairs", [1, 7, 30])
def test_pair_forms_with_fewer_pairs_than_slots(mxq, pairs):
    """The many-token launches with their grid capped below the device's
    cluster slots (a host-side launch parameter): every pair then walks more
    units and the quantising launch deals its jobs over fewer pairs; no wait
    may run out (the fixture checks the watchdog) and the outputs must be
    bit-identical to the uncapped quantiser + GEMM."""
    T, G, D, N = 1100, 8, 4096, 1024
    x, pos, cos, sin = wo_a_inputs(T, G, D, N, 64, seed=2300, pos_mode="arange")
    w, sw = oracle_weights(G, N, D, seed=3)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, D)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, 64)
    ref = mxq.mxq_bmm_a8w8(q, sc, wd, wsf)
    torch.cuda.synchronize()
    prev = mxq.mxq_debug_set_pair_limit(pairs)
    mxq.mxq_debug_takeovers(clear=True)
    try:
        out = mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=64)
        gemm = mxq.mxq_bmm_a8w8(q, sc, wd, wsf)
        torch.cuda.synchronize()
    finally:
        mxq.mxq_debug_set_pair_limit(prev)
    assert torch.equal(out, ref)
    assert torch.equal(gemm, ref)
    if pairs > 1:
        # Every pair quantises its own jobs in time: the quantisation runs
        # ahead of each pair's GEMM by enough units that the jobs a waiting
        # pair needs are always allowed.  (A single pair quantises four units'
        # jobs before its first multiply can start, which may exceed the
        # takeover wait.)
        assert mxq.mxq_debug_takeovers() == 0


@pytest.mark.parametrize("lazy_from", [0, 5, 40])
def test_pair_quant_when_owners_do_not_quantise(mxq, lazy_from):
    """Pairs of the one-launch prefill from index `lazy_from` on skip the
    quantisation jobs they own, as if they never ran (0: no pair quantises
    anything).  The pairs waiting on those jobs must quantise them
    themselves after their takeover wait -- several consumers may do the
    same job, writing the same bytes -- with no wait running out (the
    fixture checks the watchdog), and the output must be bit-identical to
    quantiser + GEMM."""
    T, G, D, N = 1100, 8, 4096, 1024
    x, pos, cos, sin = wo_a_inputs(T, G, D, N, 64, seed=2400, pos_mode="arange")
    w, sw = oracle_weights(G, N, D, seed=3)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, D)
    q, sc = mxq.mxq_inv_rope_group_quant(xd, pd, cd, sd, 64)
    ref = mxq.mxq_bmm_a8w8(q, sc, wd, wsf)
    ws = torch.full((mxq.mxq_wo_a_workspace_bytes(T, G, D, N),), 0xA5, dtype=torch.uint8,
                    device="cuda")
    torch.cuda.synchronize()
    prev = mxq.mxq_debug_set_lazy_pairs(lazy_from)
    mxq.mxq_debug_takeovers(clear=True)
    try:
        out = mxq.mxq_wo_a(xd, pd, cd, sd, wd, wsf, R=64, ws=ws)
        torch.cuda.synchronize()
    finally:
        mxq.mxq_debug_set_lazy_pairs(prev)
    assert torch.equal(out, ref)
    assert mxq.mxq_debug_takeovers() > 0  # the takeover path ran
    assert np.array_equal(ws[:T * G * D].cpu().numpy().reshape(T, G, D), q.cpu().numpy())


def test_pair_quant_takeover_with_invalid_positions(mxq):
    """Every job quantised by its consumers (no pair quantises its own), with
    some positions outside the table: those tokens' outputs are zero and the
    error bit is set, every other token as the oracle."""
    T, G, D, N = 300, 2, 512, 256
    x, _, cos, sin = wo_a_inputs(T, G, D, N, 64, seed=2500, max_pos=100, max_pos_table=100)
    rng = np.random.Generator(np.random.PCG64(2501))
    pos = torch.from_numpy(rng.integers(0, 100, T).astype(np.int64))
    bad = np.array([0, 17, 130, 255, 299])
    pos[bad] = torch.tensor([-1, 100, 1000, -7, 100], dtype=torch.int64)
    w, sw = oracle_weights(G, N, D, seed=2502)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = mxq.mxq_debug_set_lazy_pairs(0)
    try:
        out, _ = run(mxq, x, pos, cos, sin, w, sw, 64, err=err)
    finally:
        mxq.mxq_debug_set_lazy_pairs(prev)
    assert int(err.item()) == mxq.MXQ_DEVERR_POSITION
    o = out.float().cpu()
    assert (o[bad] == 0).all()
    good = np.setdiff1d(np.arange(T), bad)
    a, sa = oracle_quant(x[good], pos[good], cos, sin, 64)
    check_gemm(out[good], *O.bmm_a8w8_ref(a, sa, w, sw), "good rows, jobs taken over")
