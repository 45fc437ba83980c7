"""GPU parity of mxq_linear, the MXFP8 linear for any K (including
K % 128 != 0), against the oracle (activation group quantisation, then the
block-scaled GEMM)."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import check_gemm, oracle_weights, to_dev
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


@pytest.mark.parametrize("K", [576, 288, 2304])
@pytest.mark.parametrize("M", [1, 8])
def test_unaligned_k_linear(mxq, M, K):
    """x [M, K] ~ N(0,1) BF16, W [5120, K] from N(0, 0.02)."""
    x = W.bf16_normal((M, K), seed=3000 + M + K)
    w, sw = oracle_weights(1, 5120, K, seed=3100 + K)
    xd, wd, swd = to_dev(x, w[0], sw)
    wsf = mxq.mxq_prepare_weight_scales(swd, K)
    out = mxq.mxq_linear(xd, wd, wsf)
    torch.cuda.synchronize()
    y_ref, S, _, _ = O.linear_ref(W.bf16_bits(x), w[0], sw[0])
    check_gemm(out, y_ref, S, f"linear M={M} K={K}")


@pytest.mark.parametrize("M", [100, 130, 1000])
def test_linear_many_rows(mxq, M):
    """Quantiser + GEMM (M = 100) and one launch of the quantising CTA-pair
    GEMM (M > 128), K = 576 with its 64-wide last group."""
    K = 576
    x = W.bf16_normal((M, K), seed=3200 + M)
    w, sw = oracle_weights(1, 512, K, seed=3300)
    xd, wd, swd = to_dev(x, w[0], sw)
    out = mxq.mxq_linear(xd, wd, mxq.mxq_prepare_weight_scales(swd, K))
    torch.cuda.synchronize()
    y_ref, S, _, _ = O.linear_ref(W.bf16_bits(x), w[0], sw[0])
    check_gemm(out, y_ref, S, f"linear M={M}")


def test_linear_close_to_bf16_dequant_path(mxq):
    """Loose check against the BF16 path the dequantise-once page describes:
    BF16 x times the dequantised weight (cuBLAS here, as a reference only)."""
    M, K, N = 8, 576, 5120
    x = W.bf16_normal((M, K), seed=3400)
    w, sw = oracle_weights(1, N, K, seed=3401)
    xd, wd, swd = to_dev(x, w[0], sw)
    out = mxq.mxq_linear(xd, wd, mxq.mxq_prepare_weight_scales(swd, K)).float()
    w_bf16 = mxq.mxq_dequant_bf16(wd[None], swd)[0]
    ref = (xd.double() @ w_bf16.double().T)
    bound = (xd.double().abs() * 2.0 ** -4) @ w_bf16.double().abs().T + 1e-3
    assert bool(((out.double() - ref).abs() <= bound).all())


@pytest.mark.parametrize("M", [1, 100, 200])
def test_maximum_k_linear(mxq, M):
    """K = 65536, the largest K the ABI accepts, in each of the three launch
    forms (fused, quantiser + GEMM, quantising CTA pair)."""
    K = 65536
    x = W.bf16_normal((M, K), seed=3500 + M)
    w, sw = oracle_weights(1, 32, K, seed=3501)
    xd, wd, swd = to_dev(x, w[0], sw)
    out = mxq.mxq_linear(xd, wd, mxq.mxq_prepare_weight_scales(swd, K))
    torch.cuda.synchronize()
    y_ref, S, _, _ = O.linear_ref(W.bf16_bits(x), w[0], sw[0])
    check_gemm(out, y_ref, S, f"linear M={M} K=65536")
