"""GPU parity of the load-time kernels: MXFP8 -> BF16 dequantisation
(bit-exact), the prepared weight-scale layout, and FP32 -> E8M0 scale
conversion."""

import numpy as np
import pytest
import torch

import workloads as W
from cases import oracle_weights, to_dev
from oracle import mx_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mxq():
    import mxfp8_block_scaled_inv_gb300 as m
    from mxfp8_block_scaled_inv_gb300 import build

    build.build()
    m.lib()
    return m


def _nan_aware_equal(got, ref):
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    nan_r = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x7F) != 0)
    return np.array_equal(nan_g, nan_r) and np.array_equal(got[~nan_r], ref[~nan_r])


def test_exhaustive_code_scale_pairs(mxq):
    """Every (E4M3 code, E8M0 byte) pair: row r uses scale byte r, column k holds code k % 256."""
    codes = np.tile(np.arange(256, dtype=np.uint8), (256, 1))[None]  # [1, 256, 256]
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 2, axis=1)[None]  # [1, 256, 2]
    wd, sd = to_dev(codes, scales)
    out = mxq.mxq_dequant_bf16(wd, sd)
    torch.cuda.synchronize()
    got = W.bf16_bits(out.cpu())
    assert _nan_aware_equal(got, O.dequant_bf16(codes, scales))


@pytest.mark.parametrize("K", [576, 288, 2304])
def test_unaligned_k_production_shapes(mxq, K):
    """The DeepSeek-V4.1 shared-expert down_proj shapes (5120, K) at TP4/TP8
    and the aligned control."""
    codes, scales = oracle_weights(1, 5120, K, seed=2000 + K)
    wd, sd = to_dev(codes, scales)
    out = mxq.mxq_dequant_bf16(wd, sd)
    torch.cuda.synchronize()
    assert np.array_equal(W.bf16_bits(out.cpu()), O.dequant_bf16(codes, scales))


def test_prepared_scale_layout(mxq):
    """Byte-level check of the documented atom layout."""
    B, N, K = 2, 300, 400  # N not a multiple of 128 or 256, partial last K group
    KG = 4
    rng = np.random.Generator(np.random.PCG64(9))
    sc = rng.integers(0, 255, size=(B, N, KG), dtype=np.uint8)
    (sd,) = to_dev(sc)
    prep = mxq.mxq_prepare_weight_scales(sd, K).cpu().numpy()
    NB = 4  # rows padded to 512 -> 4 blocks of 128
    assert prep.size == B * KG * NB * 512
    atoms = prep.reshape(B, KG, NB, 32, 4, 4)  # [b, kg, nb, i, j, byte]
    for b in range(B):
        for kg in range(KG):
            for nb in range(NB):
                for j in range(4):
                    rows = nb * 128 + 32 * j + np.arange(32)
                    exp = np.where(rows < N, sc[b, np.minimum(rows, N - 1), kg], 127)
                    for byte in range(4):
                        assert np.array_equal(atoms[b, kg, nb, :, j, byte], exp)


def test_scales_f32_to_e8m0(mxq):
    ks = np.arange(-127, 128)
    good = np.ldexp(np.ones(ks.shape), ks).astype(np.float32)
    bad = np.array([0.0, -1.0, 3.0, 0.75, np.inf, -np.inf, np.nan, 2.0 ** -128, 2.0 ** -149, -0.0],
                   dtype=np.float32)
    s = np.concatenate([good, bad])
    ref, ok = O.scales_f32_to_e8m0(s)
    (sd,) = to_dev(s)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mxq.mxq_scales_f32_to_e8m0(sd, err_flag=err)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)
    assert int(err.item()) == mxq.MXQ_DEVERR_SCALE
    err.zero_()
    mxq.mxq_scales_f32_to_e8m0(to_dev(good)[0], err_flag=err)
    assert int(err.item()) == 0
