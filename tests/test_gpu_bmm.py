"""GPU parity of mxq_bmm_a8w8 (and the fused wo_a sequence) against the
oracle: every output within 1 bf16 ulp of the fp64 reference plus
1e-5 * sum_k |a_k w_k|."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import check_gemm, oracle_quant, oracle_weights, to_dev, wo_a_inputs
from conftest import read_sections
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
    assert m.mxq_watchdog_read() == 0, "a bounded wait inside a kernel ran out"


def random_operands(T, G, N, K, seed):
    """Activation codes/scales from the oracle quantiser of N(0,1) BF16 rows,
    weights from the oracle quantiser of N(0, 0.02)."""
    x = W.bf16_normal((T, G, K), seed=seed)
    a, sa = O.group_quant_rows(O.bf16_bits_to_f32(W.bf16_bits(x)))
    w, sw = oracle_weights(G, N, K, seed=seed + 1)
    return a, sa, w, sw


def run_bmm(mxq, a, sa, w, sw):
    K = a.shape[-1]
    ad, sad, wd, swd = to_dev(a, sa, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, K)
    out = mxq.mxq_bmm_a8w8(ad, sad, wd, wsf)
    torch.cuda.synchronize()
    return out


def test_tiny_fused_wo_a(mxq):
    """x [16,2,256], R=64, positions 0..15, W [2,128,256] from N(0,0.02), seed 0."""
    x, pos, cos, sin = wo_a_inputs(16, 2, 256, 128, 64, seed=0, pos_mode="arange")
    w, sw = oracle_weights(2, 128, 256, seed=1)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, 256)
    out = mxq.wo_a(xd, pd, cd, sd, wd, wsf, R=64)
    torch.cuda.synchronize()
    a, sa = oracle_quant(x, pos, cos, sin, 64)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), "tiny")


def test_two_token_handworked_gemm(mxq):
    sec = read_sections("wo_a_2token_handworked.txt")
    a = np.zeros((2, 1, 128), dtype=np.uint8)
    for t, k, c in sec["codes"]:
        a[int(t), 0, int(k)] = int(c, 16)
    sa = np.array([[[int(b)]] for _, b in sec["scales"]], dtype=np.uint8)
    w = np.zeros((1, 16, 128), dtype=np.uint8)  # N padded to 16 with zero rows
    w[0, 0, :] = 0x38
    w[0, 1, 64] = 0x40
    w[0, 2, 5] = 0x38
    w[0, 2, 96] = 0xB8
    sw = np.full((1, 16, 1), 127, dtype=np.uint8)
    for n, b in sec["w_scales"]:
        sw[0, int(n), 0] = int(b)
    out = W.bf16_bits(run_bmm(mxq, a, sa, w, sw).cpu())
    for t, n, _, bits in sec["y"]:
        assert out[int(t), 0, int(n)] == int(bits, 16)
    assert (out[:, 0, 3:] == 0).all()


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_shapes(mxq, T):
    """wo_a decode: x [T, 8, 4096] at random positions, W [8, 1024, 4096]."""
    x, pos, cos, sin = wo_a_inputs(T, 8, 4096, 1024, 64, seed=300 + T, max_pos_table=32768)
    w, sw = oracle_weights(8, 1024, 4096, seed=3)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, 4096)
    out = mxq.wo_a(xd, pd, cd, sd, wd, wsf, R=64)
    torch.cuda.synchronize()
    a, sa = oracle_quant(x, pos, cos, sin, 64)
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), f"decode T={T}")


@pytest.mark.parametrize("T", [2, 17, 100, 128, 129, 300, 517])
def test_token_counts_span_both_orientations(mxq, T):
    a, sa, w, sw = random_operands(T, 3, 512, 640, seed=800 + T)
    check_gemm(run_bmm(mxq, a, sa, w, sw), *O.bmm_a8w8_ref(a, sa, w, sw), f"T={T}")


@pytest.mark.parametrize("K", [16, 48, 160, 288, 576, 2304])
@pytest.mark.parametrize("T", [8, 200])
def test_unaligned_k(mxq, K, T):
    a, sa, w, sw = random_operands(T, 2, 256, K, seed=900 + K + T)
    check_gemm(run_bmm(mxq, a, sa, w, sw), *O.bmm_a8w8_ref(a, sa, w, sw), f"K={K} T={T}")


@pytest.mark.parametrize("N", [16, 48, 272, 1040])
@pytest.mark.parametrize("T", [5, 260])
def test_ragged_n(mxq, N, T):
    a, sa, w, sw = random_operands(T, 2, N, 384, seed=1000 + N + T)
    check_gemm(run_bmm(mxq, a, sa, w, sw), *O.bmm_a8w8_ref(a, sa, w, sw), f"N={N} T={T}")


def test_prefill_chunk_sampled(mxq):
    """One 8K prefill chunk: x [8192, 8, 4096] with 1% x50 outliers, positions
    0..8191, W [8, 1024, 4096]; checked on sampled tokens (all groups, all n)."""
    T = 8192
    x, pos, cos, sin = wo_a_inputs(T, 8, 4096, 1024, 64, seed=400, pos_mode="arange",
                                   outlier_frac=0.01)
    w, sw = oracle_weights(8, 1024, 4096, seed=3)
    xd, pd, cd, sd, wd, swd = to_dev(x, pos, cos, sin, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, 4096)
    out = mxq.wo_a(xd, pd, cd, sd, wd, wsf, R=64)
    torch.cuda.synchronize()
    rng = np.random.Generator(np.random.PCG64(402))
    idx = np.unique(np.concatenate([[0, 127, 128, T - 1], rng.integers(0, T, 60)]))
    a, sa = oracle_quant(x[idx], pos[idx], cos, sin, 64)
    check_gemm(out[idx], *O.bmm_a8w8_ref(a, sa, w, sw), "prefill sampled")


def test_deterministic(mxq):
    a, sa, w, sw = random_operands(32, 8, 1024, 4096, seed=1100)
    o1 = run_bmm(mxq, a, sa, w, sw)
    o2 = run_bmm(mxq, a, sa, w, sw)
    assert torch.equal(o1, o2)


def test_empty_tokens_is_noop(mxq):
    a = torch.empty((0, 2, 256), dtype=torch.uint8, device="cuda")
    sa = torch.empty((0, 2, 2), dtype=torch.uint8, device="cuda")
    w, sw = oracle_weights(2, 128, 256, seed=5)
    wd, swd = to_dev(w, sw)
    out = mxq.mxq_bmm_a8w8(a, sa, wd, mxq.mxq_prepare_weight_scales(swd, 256))
    assert out.shape == (0, 2, 128)


@pytest.mark.parametrize("T,G,N,K", [(257, 1, 16, 256), (257, 2, 48, 384), (384, 1, 272, 2304),
                                     (1000, 3, 1040, 640)])
def test_pair_form_edges(mxq, T, G, N, K):
    """Many-token (CTA-pair) form at its edges: the odd CTA's 128 tokens partly
    or wholly past T (T = 257, 384), weight tiles mostly past N (N = 16, 48,
    272, 1040), one group, unaligned K; TMA clips the output stores."""
    a, sa, w, sw = random_operands(T, G, N, K, seed=1200 + T + N)
    check_gemm(run_bmm(mxq, a, sa, w, sw), *O.bmm_a8w8_ref(a, sa, w, sw), f"pair T={T} N={N}")


def test_pair_form_deterministic(mxq):
    a, sa, w, sw = random_operands(600, 4, 512, 1024, seed=1300)
    o1 = run_bmm(mxq, a, sa, w, sw)
    o2 = run_bmm(mxq, a, sa, w, sw)
    assert torch.equal(o1, o2)


def test_pair_form_leaves_padding_untouched(mxq):
    """Rows past T and columns past N are not written by the clipped stores:
    out is a view into a larger buffer whose surroundings stay intact."""
    T, G, N, K = 300, 2, 48, 256
    a, sa, w, sw = random_operands(T, G, N, K, seed=1400)
    ad, sad, wd, swd = to_dev(a, sa, w, sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, K)
    big = torch.full((T + 5, G, N), -7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:T]
    mxq.mxq_bmm_a8w8(ad, sad, wd, wsf, out=out)
    torch.cuda.synchronize()
    assert bool((big[T:] == -7.0).all())
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), "pair padding")


@pytest.mark.parametrize("T", [5, 257])
def test_maximum_k(mxq, T):
    """K = 65536, the largest K the ABI accepts (512 scale groups): the
    few-token form splits it over a cluster of 8 CTAs, the pair form runs all
    512 groups through one accumulator."""
    a, sa, w, sw = random_operands(T, 1, 16, 65536, seed=1500 + T)
    check_gemm(run_bmm(mxq, a, sa, w, sw), *O.bmm_a8w8_ref(a, sa, w, sw), f"K=65536 T={T}")


def _random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38  # no NaN codes
    return c


@pytest.mark.parametrize("T", [2, 129])
def test_maximum_groups(mxq, T):
    """G = 65535, the largest batch the ABI accepts, in the few-token and the
    pair form (random codes and scale bytes; sampled tokens for the pair form)."""
    G, N, K = 65535, 16, 128
    rng = np.random.Generator(np.random.PCG64(1600 + T))
    a = _random_codes(rng, (T, G, K))
    sa = rng.integers(118, 136, size=(T, G, 1), dtype=np.uint8)
    w = _random_codes(rng, (G, N, K))
    sw = rng.integers(118, 136, size=(G, N, 1), dtype=np.uint8)
    out = run_bmm(mxq, a, sa, w, sw)
    idx = np.arange(T) if T <= 4 else np.array([0, 127, 128, T - 1])
    check_gemm(out[torch.from_numpy(idx).to(out.device)], *O.bmm_a8w8_ref(a[idx], sa[idx], w, sw),
               f"G=65535 T={T}")
