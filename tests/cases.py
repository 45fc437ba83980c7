"""Shared helpers of the GPU parity tests: seeded inputs (from workloads),
oracle references (from oracle), and the comparison rules."""

import functools

import numpy as np
import torch

import workloads as W
from oracle import mx_oracle as O

DEV = "cuda"


def wo_a_inputs(T, G, D, N, R, seed, max_pos=32768, pos_mode="uniform", outlier_frac=0.0,
                max_pos_table=None):
    """x bf16 [T,G,D], pos int64 [T], cos/sin bf16 [max_pos, R/2], FP32 weights -> oracle codes."""
    x = W.bf16_normal((T, G, D), seed=seed, outlier_frac=outlier_frac)
    if pos_mode == "arange":
        pos = W.positions_arange(0, T)
    else:
        pos = W.positions_uniform(T, seed=seed + 1, max_pos=max_pos)
    table_rows = max_pos_table or max(int(pos.max()) + 1 if T > 0 else 1, 1)
    cos, sin = W.rope_cache(table_rows, max(R, 2))
    return x, pos, cos, sin


@functools.lru_cache(maxsize=8)
def oracle_weights(G, N, K, seed, std=0.02):
    """Oracle E4M3 codes / E8M0 bytes of N(0, std) FP32 weights (cached; read-only)."""
    wf = W.f32_normal((G, N, K), seed=seed, std=std).numpy()
    return O.group_quant_rows(wf)


def oracle_quant(x, pos, cos, sin, R):
    return O.inv_rope_group_quant(W.bf16_bits(x), pos.numpy(), W.bf16_bits(cos),
                                  W.bf16_bits(sin), R)


def check_gemm(out_bf16, y_ref, S, what=""):
    """|y - y_ref| <= 1 bf16 ulp(y_ref) + 1e-5 * sum|a w|, element by element."""
    y = out_bf16.float().cpu().numpy().astype(np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    err = np.abs(y - y_ref)
    tol = O.gemm_tolerance(y_ref, S)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()}"
                             f" y={y[tuple(idx[0])]} ref={y_ref[tuple(idx[0])]} tol={tol[tuple(idx[0])]}")
    return float(np.max(err / tol)) if err.size else 0.0


def to_dev(*arrs):
    out = []
    for a in arrs:
        if isinstance(a, np.ndarray):
            a = torch.from_numpy(np.ascontiguousarray(a))
        out.append(a.to(DEV))
    return out
