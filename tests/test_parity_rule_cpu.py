"""The GEMM comparison rule of the GPU parity tests, on the CPU.

check_gemm has to accept what a correct kernel can return (the exact sum
rounded once to BF16, or an fp32 accumulation of the exact products rounded
to BF16) and reject plausible kernel mistakes: an output off by two BF16
ulps, two tokens swapped, the last (partial) K group dropped, one scale
byte off by one, and the weights of the wrong batch group."""

import numpy as np
import pytest
import torch

from cases import check_gemm
from oracle import mx_oracle as O

T, G, N, K = 8, 2, 64, 288  # K = 2 full groups + a 32-wide tail


def _operands(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.integers(0, 256, size=(T, G, K), dtype=np.uint8)
    w = rng.integers(0, 256, size=(G, N, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x30
    w[(w & 0x7F) == 0x7F] = 0x30
    sa = rng.integers(120, 134, size=(T, G, 3), dtype=np.uint8)
    sw = rng.integers(120, 134, size=(G, N, 3), dtype=np.uint8)
    return a, sa, w, sw


def _bf16(y):
    bits = O.bf16_rne_bits(y).astype(np.int16)
    return torch.from_numpy(bits).view(torch.bfloat16)


@pytest.fixture(scope="module")
def ref():
    a, sa, w, sw = _operands(51)
    y, S = O.bmm_a8w8_ref(a, sa, w, sw)
    return a, sa, w, sw, y, S


def test_accepts_the_exact_sum_rounded_once(ref):
    *_, y, S = ref
    assert check_gemm(_bf16(y), y, S) <= 0.5 + 1e-12  # half an ulp at most


def test_accepts_fp32_accumulation(ref):
    a, sa, w, sw, y, S = ref
    A = O.mx_values(a, sa).astype(np.float32)
    Wv = O.mx_values(w, sw).astype(np.float32)
    acc = np.zeros((T, G, N), dtype=np.float32)
    for k in range(K):  # products are exact in fp32 here; the running sum rounds
        acc += A[:, :, None, k] * Wv[None, :, :, k].astype(np.float32)
    check_gemm(_bf16(acc.astype(np.float64)), y, S)


def test_rejects_two_ulp_error(ref):
    *_, y, S = ref
    out = _bf16(y).view(torch.int16).clone()
    big = np.unravel_index(np.argmax(np.abs(y)), y.shape)
    out[big] += 2
    with pytest.raises(AssertionError):
        check_gemm(out.view(torch.bfloat16), y, S)


def test_rejects_swapped_tokens(ref):
    *_, y, S = ref
    out = _bf16(y).clone()
    out[[0, 1]] = out[[1, 0]]
    with pytest.raises(AssertionError):
        check_gemm(out, y, S)


def test_rejects_dropped_tail_group(ref):
    a, sa, w, sw, y, S = ref
    a2 = a.copy()
    a2[..., 256:] = 0
    y2, _ = O.bmm_a8w8_ref(a2, sa, w, sw)
    with pytest.raises(AssertionError):
        check_gemm(_bf16(y2), y, S)


def test_rejects_scale_off_by_one(ref):
    a, sa, w, sw, y, S = ref
    sw2 = sw.copy()
    sw2[:, :, 1] += 1
    y2, _ = O.bmm_a8w8_ref(a, sa, w, sw2)
    with pytest.raises(AssertionError):
        check_gemm(_bf16(y2), y, S)


def test_rejects_weights_of_the_wrong_group(ref):
    a, sa, w, sw, y, S = ref
    y2, _ = O.bmm_a8w8_ref(a, sa, w[::-1].copy(), sw[::-1].copy())
    with pytest.raises(AssertionError):
        check_gemm(_bf16(y2), y, S)
