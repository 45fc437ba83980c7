"""mxq_linear_noalloc: the MXFP8 linear for callers that cannot allocate
device memory (a plain-C host program with no device allocator of its own,
or a serving loop that must not call cudaMalloc/cudaFree because they can
synchronise the device).  It runs the same kernels as mxq_linear but takes
its scratch from a fixed array inside the library.

This file is collected last on purpose: the entry point shares one array
per device across calls, so it is also exercised after every other test has
run in the same process; it must pass both ways."""

import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from cases import check_gemm, oracle_weights, to_dev
from oracle import mx_oracle as O


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    return m


def _noalloc(mxq, x, w, wsf):
    """Call the entry point through the C ABI (ctypes), on the current stream."""
    M, K = x.shape
    N = w.shape[0]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = mxq.lib().mxq_linear_noalloc(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(wsf.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), M, N, K,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, mxq.lib().mxq_last_error()
    return out


# (M, K, seed): two calls in a row share the array (larger, then smaller
# problem, other inputs); M = 8 and 3 take the single fused launch, which
# needs no scratch; M = 100 and 7219 go through the array, and 7219 rows at
# K = 576 (4,158,144 code bytes + 36,095 scale bytes, each rounded up to 256)
# fill it to its last byte.
CASES = [(8, 2304, 4100), (3, 576, 4200), (100, 2304, 4300), (7219, 576, 4400), (40, 576, 4500)]


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_linear_on_calls_in_a_row(mxq):
    N = 5120
    for M, K, seed in CASES:
        x = W.bf16_normal((M, K), seed=seed)
        w, sw = oracle_weights(1, N, K, seed=seed + 1)
        xd, wd, swd = to_dev(x, w[0], sw)
        wsf = mxq.mxq_prepare_weight_scales(swd, K)
        got = _noalloc(mxq, xd, wd, wsf)
        ref = mxq.mxq_linear(xd, wd, wsf)
        torch.cuda.synchronize()
        # Against the oracle (activation group quantisation, then the fp64
        # block-scaled GEMM), at the GEMM parity tolerance.
        y_ref, S, _, _ = O.linear_ref(W.bf16_bits(x), w[0], sw[0])
        check_gemm(got, y_ref, S, f"noalloc M={M} K={K}")
        # And against the entry point with a caller workspace, within the same tolerance.
        g = got.float().cpu().numpy().astype(np.float64)
        r = ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(g - r) <= O.gemm_tolerance(y_ref, S)), f"M={M} K={K}"


def test_noalloc_rejects_sizes_beyond_the_scratch():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    L = m.lib()
    p = ctypes.c_void_p(1 << 20)
    # 7220 rows at K = 576 need 4,195,072 bytes > 4 MiB: rejected before any launch.
    assert L.mxq_linear_noalloc(p, p, p, p, 7220, 5120, 576, None) == 6
    assert b"scratch" in L.mxq_last_error()
    assert L.mxq_linear_noalloc(p, p, p, p, 4, 5120, 570, None) == 2
    assert L.mxq_linear_noalloc(p, p, p, p, 0, 5120, 576, None) == 0
    # Every rule of mxq_linear is checked before anything is enqueued (without
    # a GPU, a call that got as far as a launch would report a CUDA or
    # architecture error instead of these).
    u = ctypes.c_void_p((1 << 20) + 8)
    assert L.mxq_linear_noalloc(p, p, p, u, 100, 5120, 576, None) == 3  # misaligned out
    assert L.mxq_linear_noalloc(p, p, u, p, 1, 5120, 576, None) == 3    # misaligned scales
    assert L.mxq_linear_noalloc(p, u, p, p, 40, 5120, 576, None) == 3   # misaligned weight
    assert L.mxq_linear_noalloc(p, p, p, p, 1, 5120, 131072, None) == 4  # K > 65536
    assert L.mxq_linear_noalloc(p, p, p, p, 0, 5120, 131072, None) == 4  # checked before M == 0
    assert L.mxq_linear_noalloc(p, p, p, p, 1, 1 << 25, 65536, None) == 4  # N*K >= 2^40
    assert L.mxq_linear_noalloc(p, p, p, None, 1, 5120, 576, None) == 1
