"""GPU parity of the 100,000-token prefill stream: one 100K prompt prefilled
in 8K chunks (page "[ROCm][DSV4][Perf] Use FP8 WO_A output projection",
Performance: the TTFT of a 100K-token prompt, chunked at 8192 tokens), i.e.
12 chunks of 8192 tokens and a last chunk of 1696 at positions 98,304..99,999,
each through mxq_wo_a with the production shapes G = 8, D = K = 4096,
N = 1024, R = 64 and a cos/sin cache of 100,000 rows.

The last chunk is checked whole: every code and scale byte the one-launch
prefill writes to its workspace (bit-exact), and every output element
against the oracle at the GEMM tolerance.  Its last 256-token block holds
only 160 tokens, so the odd CTA of the last pair has 32 rows and the rest
of the pair's tiles lie past T.  Two full 8K chunks at positions >= 32,768
(chunks 4 and 11 of the stream) are checked on sampled tokens: the first and
last token of 128-token blocks, and random ones."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import check_gemm, oracle_quant, oracle_weights, to_dev
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu

G, D, N, R = 8, 4096, 1024, 64
MAX_POS = 100000


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    m.mxq_watchdog_read(clear=True)
    yield m
    assert m.mxq_watchdog_read() == 0


@pytest.fixture(scope="module")
def stream_state(mxq):
    cos, sin = W.rope_cache(MAX_POS, R)
    w, sw = oracle_weights(G, N, D, seed=3)
    cd, sd, wd, swd = to_dev(cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, D)
    ws = torch.empty(mxq.mxq_wo_a_workspace_bytes(8192, G, D, N), dtype=torch.uint8, device="cuda")
    return dict(cos=cos, sin=sin, w=w, sw=sw, cd=cd, sd=sd, wd=wd, wsf=wsf, ws=ws)


def run_chunk(mxq, st, chunk, T, start):
    x = W.bf16_normal((T, G, D), seed=9500 + chunk, outlier_frac=0.01)
    pos = W.positions_arange(start, T)
    xd, pd = to_dev(x, pos)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mxq.mxq_debug_takeovers(clear=True)
    out = mxq.mxq_wo_a(xd, pd, st["cd"], st["sd"], st["wd"], st["wsf"], R=R, err_flag=err,
                       ws=st["ws"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # With every pair resident, each quantises its own jobs in time.
    assert mxq.mxq_debug_takeovers() == 0
    return x, pos, out


def atom_scales(ws, T):
    """Scale bytes [T, G, KG] read back from the workspace's scale atoms."""
    r256 = lambda v: (v + 255) // 256 * 256
    MB = 2 * ((T + 255) // 256)
    KG = D // 128
    atoms = r256(T * G * D)
    at = ws[atoms:atoms + G * MB * KG * 512].cpu().numpy().reshape(G, MB, KG, 32, 4, 4)
    assert (at == at[..., :1]).all(), "an atom word does not repeat its byte"
    b = at[..., 0].transpose(0, 1, 4, 3, 2).reshape(G, MB * 128, KG)
    assert (b[:, T:, :] == 127).all(), "rows past the chunk must hold byte 127"
    return b[:, :T, :].transpose(1, 0, 2)


def test_last_chunk_1696_tokens_whole(mxq, stream_state):
    st = stream_state
    T, start = 1696, 12 * 8192
    x, pos, out = run_chunk(mxq, st, 12, T, start)
    assert int(pos[-1]) == MAX_POS - 1
    a, sa = oracle_quant(x, pos, st["cos"], st["sin"], R)
    codes = st["ws"][:T * G * D].cpu().numpy().reshape(T, G, D)
    assert np.array_equal(codes, a), "codes differ from the oracle"
    assert np.array_equal(atom_scales(st["ws"], T), sa), "scale bytes differ from the oracle"
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, st["w"], st["sw"]), "100K stream, chunk of 1696")


@pytest.mark.parametrize("chunk", [4, 11])
def test_full_chunks_at_high_positions_sampled(mxq, stream_state, chunk):
    st = stream_state
    T, start = 8192, chunk * 8192
    assert start >= 32768
    x, pos, out = run_chunk(mxq, st, chunk, T, start)
    rng = np.random.Generator(np.random.PCG64(9600 + chunk))
    edges = np.concatenate([np.arange(0, T, 128 * 7), np.arange(127, T, 128 * 9), [T - 1]])
    idx = np.unique(np.concatenate([edges, rng.integers(0, T, 24)]))
    a, sa = oracle_quant(x[idx], pos[idx], st["cos"], st["sin"], R)
    check_gemm(out[idx], *O.bmm_a8w8_ref(a, sa, st["w"], st["sw"]),
               f"100K stream, chunk {chunk} (positions {start}..{start + T - 1}), sampled tokens")
