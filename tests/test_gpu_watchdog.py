"""The bounded-wait failure path, exercised without faulting the GPU: a
kernel waits on a barrier nothing completes, gives up after its limit, sets
the watchdog word and returns; the context keeps working afterwards."""

import pytest
import torch

from cases import check_gemm, oracle_weights, to_dev
import workloads as W
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    return m


def test_wait_that_runs_out_reports_and_returns(mxq):
    mxq.mxq_watchdog_read(clear=True)
    mxq.mxq_watchdog_selftest(limit_ns=2_000_000)  # 2 ms
    torch.cuda.synchronize()  # returns: the kernel gave up instead of hanging
    assert mxq.mxq_watchdog_read(clear=True) == 1 << 31
    assert mxq.mxq_watchdog_read() == 0
    # The context is intact: a GEMM right after still matches the oracle.
    x = W.bf16_normal((4, 1, 256), seed=77)
    a, sa = O.group_quant_rows(O.bf16_bits_to_f32(W.bf16_bits(x)))
    w, sw = oracle_weights(1, 128, 256, seed=78)
    ad, sad, wd, swd = to_dev(a, sa, w, sw)
    out = mxq.mxq_bmm_a8w8(ad, sad, wd, mxq.mxq_prepare_weight_scales(swd, 256))
    torch.cuda.synchronize()
    check_gemm(out, *O.bmm_a8w8_ref(a, sa, w, sw), "after watchdog")
    assert mxq.mxq_watchdog_read() == 0


def test_selftest_limit_is_validated(mxq):
    with pytest.raises(mxq.MxqError):
        mxq.mxq_watchdog_selftest(limit_ns=0)
    with pytest.raises(mxq.MxqError):
        mxq.mxq_watchdog_selftest(limit_ns=3_000_000_000)
