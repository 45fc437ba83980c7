"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects invalid arguments on the host (returning the
documented status and launching nothing)."""

import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mxq.h")


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_inv_gb300 import build as B

    B.build()
    import mxfp8_block_scaled_inv_gb300 as mxq

    return mxq.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["mxq_inv_rope_group_quant", "mxq_bmm_a8w8", "mxq_linear", "mxq_dequant_bf16",
              "mxq_prepare_weight_scales", "mxq_scales_f32_to_e8m0"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.mxq_status_string(0) == b"MXQ_OK"
    assert L.mxq_status_string(5) == b"MXQ_ERR_ARCH"
    assert L.mxq_status_string(99) == b"MXQ_ERR_UNKNOWN"
    assert L.mxq_version() >= 100


def test_arch_gate(L):
    assert L.mxq_arch_supported(10, 3) == 1
    for mm in [(10, 0), (10, 1), (9, 0), (12, 0), (8, 9)]:
        assert L.mxq_arch_supported(*mm) == 0


P = ctypes.c_void_p(1 << 20)     # 16-byte aligned fake device address (never dereferenced)
U = ctypes.c_void_p((1 << 20) + 8)  # misaligned


def quant(L, x=P, T=4, G=1, D=256, R=0, pos=P, cos=P, sin=P, cs_ld=32, max_pos=16, q=P, sc=P,
          err=None):
    return L.mxq_inv_rope_group_quant(x, T, G, D, R, pos, cos, sin, cs_ld, max_pos, q, sc, err, None)


def test_quant_argument_errors(L):
    assert quant(L, x=None) == 1
    assert quant(L, q=None) == 1
    assert quant(L, T=-1) == 2
    assert quant(L, G=0) == 2
    assert quant(L, D=8) == 2
    assert quant(L, D=264) == 2                 # D % 16
    assert quant(L, R=8, D=256) == 4            # R % 16
    assert quant(L, R=144, D=256) == 4          # R > 128
    assert quant(L, R=64, D=272) == 4           # RoPE needs D % 128 == 0
    assert quant(L, R=64, cs_ld=16) == 2        # cs_ld < R/2
    assert quant(L, R=64, cs_ld=36) == 3        # cs_ld % 8
    assert quant(L, R=64, max_pos=0) == 2
    assert quant(L, R=64, pos=None) == 1
    assert quant(L, x=U) == 3
    assert quant(L, R=64, cos=U) == 3
    assert quant(L, err=ctypes.c_void_p((1 << 20) + 2)) == 3
    assert quant(L, T=0, x=None, q=None, sc=None) == 0  # empty input is a no-op
    # sizes past the 32-bit index range: rejected before any product can overflow
    assert quant(L, T=1 << 31) == 4
    assert quant(L, T=1 << 40, G=1 << 30) == 4
    assert quant(L, T=1 << 20, G=1 << 9, D=512) == 4      # T*G*KG = 2^31
    assert quant(L, T=1 << 20, G=1 << 11, D=256) == 4     # T*G = 2^31
    assert quant(L, T=(1 << 62), G=(1 << 31) - 1) == 4


def bmm(L, a=P, asf=P, w=P, wsf=P, out=P, T=4, G=1, N=128, K=256, ws=None, ws_bytes=0):
    return L.mxq_bmm_a8w8(a, asf, w, wsf, out, T, G, N, K, ws, ws_bytes, None)


def test_bmm_argument_errors(L):
    assert bmm(L, a=None) == 1
    assert bmm(L, wsf=None) == 1
    assert bmm(L, K=8) == 2
    assert bmm(L, K=264) == 2
    assert bmm(L, N=120) == 2
    assert bmm(L, G=0) == 2
    assert bmm(L, T=-3) == 2
    assert bmm(L, K=65536 + 16) == 4
    assert bmm(L, out=U) == 3
    assert bmm(L, T=0, a=None, out=None) == 0
    assert bmm(L, T=1 << 31) == 4
    assert bmm(L, G=65536) == 4
    assert bmm(L, N=1 << 25, K=1 << 16) == 4                # N*K = 2^41
    assert L.mxq_bmm_workspace_bytes(8192, 8, 1024, 4096) == 0


def test_linear_argument_errors(L):
    assert L.mxq_linear_workspace_bytes(8, 5120, 576) == 0  # <= 32 rows: one fused launch
    need = L.mxq_linear_workspace_bytes(100, 5120, 576)
    assert need == 100 * 576 + 512  # codes (57600 B, 256-aligned) + 100*5 scale bytes -> 512
    # Above 128 rows: one launch, the workspace of mxq_wo_a with G = 1.
    assert L.mxq_linear_workspace_bytes(300, 5120, 576) == L.mxq_wo_a_workspace_bytes(300, 1, 576, 5120)
    assert L.mxq_linear(P, P, P, P, 100, 5120, 576, None, 0, None) == 6
    assert L.mxq_linear(P, P, P, P, 100, 5120, 576, P, need - 1, None) == 6
    assert L.mxq_linear(None, P, P, P, 8, 5120, 576, P, need, None) == 1
    assert L.mxq_linear(P, P, P, P, 8, 5120, 570, P, need, None) == 2
    assert L.mxq_linear(P, P, P, P, 0, 5120, 576, None, 0, None) == 0
    assert L.mxq_linear(P, P, P, P, 1 << 31, 5120, 576, P, 1 << 62, None) == 4
    assert L.mxq_linear(P, P, P, P, 1 << 62, 5120, 576, P, 1 << 62, None) == 4
    assert L.mxq_linear(P, P, P, P, 8, 1 << 25, 65536, P, 0, None) == 4   # N*K = 2^41
    assert L.mxq_linear(P, P, P, P, 8, 5120, 65536 + 16, P, 0, None) == 4


def wo_a(L, x=P, pos=P, cos=P, sin=P, cs_ld=32, max_pos=16, w=P, wsf=P, out=P, T=4, G=8, D=4096,
         N=1024, R=64, err=None, ws=None, ws_bytes=0):
    return L.mxq_wo_a(x, pos, cos, sin, cs_ld, max_pos, w, wsf, out, T, G, D, N, R, err, ws,
                      ws_bytes, None)


def test_wo_a_argument_errors(L):
    assert wo_a(L, x=None) == 1
    assert wo_a(L, pos=None) == 1
    assert wo_a(L, wsf=None) == 1
    assert wo_a(L, D=4100) == 2
    assert wo_a(L, N=1000) == 2
    assert wo_a(L, R=8) == 4
    assert wo_a(L, D=4160, R=64) == 4
    assert wo_a(L, cs_ld=36) == 3
    assert wo_a(L, out=U) == 3
    assert wo_a(L, T=0, x=None, out=None) == 0
    assert L.mxq_wo_a_workspace_bytes(32, 8, 4096, 1024) == 0
    assert L.mxq_wo_a_workspace_bytes(33, 8, 4096, 1024) == 33 * 8 * 4096 + 33 * 8 * 32
    assert L.mxq_wo_a_workspace_bytes(128, 8, 4096, 1024) == 128 * 8 * 4096 + 128 * 8 * 32
    # Above 128 tokens: codes [T, G, D], scale atoms [G, 2*ceil(T/256), ceil(D/128), 512] and
    # job counters [G, 2*ceil(T/256), ceil(D/128)] uint32, each region rounded up to 256 bytes.
    jobs = 8 * 64 * 32
    assert L.mxq_wo_a_workspace_bytes(8192, 8, 4096, 1024) == 8192 * 8 * 4096 + jobs * 512 + jobs * 4
    jobs = 3 * 6 * 5
    assert L.mxq_wo_a_workspace_bytes(700, 3, 576, 1024) == (
        (700 * 3 * 576 + 255) // 256 * 256 + jobs * 512 + (jobs * 4 + 255) // 256 * 256)
    assert wo_a(L, T=8192) == 6  # prefill sizes go through the workspace
    assert wo_a(L, T=1 << 31) == 4
    assert wo_a(L, T=1 << 62) == 4
    assert wo_a(L, G=65536) == 4
    assert wo_a(L, N=1 << 25, D=65536) == 4                 # N*D = 2^41
    assert wo_a(L, T=1 << 24, G=8, D=4096, ws=P, ws_bytes=1 << 62) == 4  # T*G*KG = 2^32


def test_dequant_and_scale_argument_errors(L):
    assert L.mxq_dequant_bf16(None, P, P, 1, 16, 128, None) == 1
    assert L.mxq_dequant_bf16(P, P, P, 1, 16, 120, None) == 2
    assert L.mxq_dequant_bf16(P, U, P, 1, 16, 128, None) == 3
    assert L.mxq_dequant_bf16(P, P, P, 0, 16, 128, None) == 0
    assert L.mxq_scales_f32_to_e8m0(None, 4, P, None, None) == 1
    assert L.mxq_scales_f32_to_e8m0(P, -1, P, None, None) == 2
    assert L.mxq_scales_f32_to_e8m0(P, 0, None, None, None) == 0
    assert L.mxq_prepare_weight_scales(P, 1, 128, 100, P, None) == 2
    assert L.mxq_prepare_weight_scales(None, 1, 128, 128, P, None) == 1


def test_weight_scale_bytes(L):
    # G * ceil(K/128) * (rows padded to 256)/128 * 512
    assert L.mxq_weight_scale_bytes(8, 1024, 4096) == 8 * 32 * 8 * 512
    assert L.mxq_weight_scale_bytes(1, 5120, 576) == 5 * 40 * 512
    assert L.mxq_weight_scale_bytes(2, 128, 256) == 2 * 2 * 2 * 512
    assert L.mxq_weight_scale_bytes(0, 128, 256) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_cuda_error(L):
    assert quant(L) == 7
    assert bmm(L) == 7


def kv_insert(L, q=P, q_out=ctypes.c_void_p(1 << 30), T=4, H=2, Dq=512, kv=P, Dk=512, pos=P, cos=P,
              sin=P, cs_ld=32, max_pos=16, R=64, slot=P, cache=P, num_slots=8, dtype=0, scale=P,
              err=None):
    return L.mxq_rope_kv_insert(q, q_out, T, H, Dq, kv, Dk, pos, cos, sin, cs_ld, max_pos, R, slot,
                                cache, num_slots, dtype, scale, err, None)


def test_rope_kv_insert_argument_errors(L):
    assert kv_insert(L, kv=None) == 1
    assert kv_insert(L, slot=None) == 1
    assert kv_insert(L, cache=None) == 1
    assert kv_insert(L, q=None) == 1
    assert kv_insert(L, scale=None) == 1                 # E4M3 cache needs its scale
    assert kv_insert(L, scale=None, dtype=1) != 1        # BF16 cache does not
    assert kv_insert(L, pos=None) == 1
    assert kv_insert(L, Dk=8) == 2
    assert kv_insert(L, Dk=520) == 2
    assert kv_insert(L, Dq=520) == 2
    assert kv_insert(L, T=-1) == 2
    assert kv_insert(L, num_slots=-1) == 2
    assert kv_insert(L, R=8) == 4
    assert kv_insert(L, R=528) == 4                      # R > Dk
    assert kv_insert(L, Dq=256, R=272, Dk=512) == 4      # R > Dq
    assert kv_insert(L, dtype=2) == 4
    assert kv_insert(L, cs_ld=36) == 3
    assert kv_insert(L, cs_ld=16) == 2
    assert kv_insert(L, kv=U) == 3
    assert kv_insert(L, q_out=U) == 3
    assert kv_insert(L, scale=ctypes.c_void_p((1 << 20) + 2)) == 3
    assert kv_insert(L, slot=ctypes.c_void_p((1 << 20) + 4)) == 3
    assert kv_insert(L, q_out=ctypes.c_void_p((1 << 20) + 1024)) == 2  # overlaps q, not q itself
    assert kv_insert(L, T=0, kv=None, cache=None, slot=None) == 0
    assert kv_insert(L, T=1 << 31) == 4
    assert kv_insert(L, T=1 << 20, H=64, Dq=512) == 4     # T*H*Dq/8 >= 2^31
    # H = 0: no query pointers needed
    assert kv_insert(L, q=None, q_out=None, H=0, Dq=0) != 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_rope_kv_insert_valid_call_without_device(L):
    assert kv_insert(L) == 7
    assert kv_insert(L, q_out=P) == 7  # in place


def test_pair_limit_is_a_plain_setting(L):
    assert L.mxq_debug_set_pair_limit(5) == 0
    assert L.mxq_debug_set_pair_limit(-3) == 5
    assert L.mxq_debug_set_pair_limit(0) == 0


def test_lazy_pairs_is_a_plain_setting(L):
    assert L.mxq_debug_set_lazy_pairs(3) == -1
    assert L.mxq_debug_set_lazy_pairs(-1) == 3
    assert L.mxq_debug_set_lazy_pairs(-5) == -1


def test_takeover_count_arguments(L):
    assert L.mxq_debug_takeovers(None, 0) == 1  # MXQ_ERR_NULL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_takeover_count_without_device(L):
    v = ctypes.c_uint32(0)
    assert L.mxq_debug_takeovers(ctypes.byref(v), 1) == 7
