"""Python binding of libmxq (the MX-scaled FP8 ``wo_a`` path for GB300).

Argument marshalling only: every function here checks nothing that the C
ABI does not check itself, allocates output tensors with torch when the
caller passes none, and forwards raw device pointers plus the current
torch CUDA stream to the entry point of the same name in ``libmxq.so``.
All arithmetic runs in the library's CUDA kernels; there is no other path.
A missing or unbuilt library raises ``MxqLibraryError`` on first use.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MxqError", "MxqLibraryError", "lib", "library_path",
    "mxq_inv_rope_group_quant", "mxq_weight_scale_bytes", "mxq_prepare_weight_scales",
    "mxq_bmm_workspace_bytes", "mxq_bmm_a8w8", "mxq_linear_workspace_bytes", "mxq_linear",
    "mxq_linear_noalloc",
    "mxq_dequant_bf16", "mxq_scales_f32_to_e8m0", "mxq_watchdog_read", "mxq_watchdog_selftest",
    "mxq_arch_supported",
    "mxq_version", "mxq_wo_a_workspace_bytes", "mxq_wo_a", "wo_a", "mxq_rope_kv_insert",
    "mxq_debug_set_pair_limit", "mxq_debug_set_lazy_pairs", "mxq_debug_takeovers",
]

HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(HERE, "libmxq.so")

MXQ_DEVERR_POSITION = 0x1
MXQ_DEVERR_SCALE = 0x2
MXQ_DEVERR_SLOT = 0x4
MXQ_CACHE_E4M3 = 0
MXQ_CACHE_BF16 = 1


class MxqLibraryError(RuntimeError):
    """libmxq.so is missing or cannot be loaded."""


class MxqError(RuntimeError):
    def __init__(self, fn, status, detail):
        self.status = status
        super().__init__(f"{fn}: {_status_name(status)}: {detail}")


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t

_SIGNATURES = {
    "mxq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mxq_last_error": (ctypes.c_char_p, []),
    "mxq_version": (ctypes.c_int, []),
    "mxq_arch_supported": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "mxq_inv_rope_group_quant": (ctypes.c_int, [_vp, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _i64,
                                                _i64, _vp, _vp, _vp, _vp]),
    "mxq_weight_scale_bytes": (_sz, [_i32, _i32, _i32]),
    "mxq_prepare_weight_scales": (ctypes.c_int, [_vp, _i32, _i32, _i32, _vp, _vp]),
    "mxq_bmm_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32]),
    "mxq_bmm_a8w8": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp, _sz, _vp]),
    "mxq_linear_workspace_bytes": (_sz, [_i64, _i32, _i32]),
    "mxq_linear": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp, _sz, _vp]),
    "mxq_dequant_bf16": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _vp]),
    "mxq_scales_f32_to_e8m0": (ctypes.c_int, [_vp, _i64, _vp, _vp, _vp]),
    "mxq_watchdog_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "mxq_linear_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp]),
    "mxq_watchdog_selftest": (ctypes.c_int, [ctypes.c_uint64, _vp]),
    "mxq_debug_set_pair_limit": (ctypes.c_int, [ctypes.c_int]),
    "mxq_debug_set_lazy_pairs": (ctypes.c_int, [ctypes.c_int]),
    "mxq_debug_takeovers": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "mxq_wo_a_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32]),
    "mxq_rope_kv_insert": (ctypes.c_int, [_vp, _vp, _i64, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _i64,
                                          _i64, _i32, _vp, _vp, _i64, _i32, _vp, _vp, _vp]),
    "mxq_wo_a": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
                                _i32, _vp, _vp, _sz, _vp]),
}


def lib():
    """The loaded ctypes library (loaded once)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise MxqLibraryError(
                f"{library_path} not found; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` or "
                "`python mxfp8_block_scaled_inv_gb300/build.py`")
        try:
            handle = ctypes.CDLL(library_path)
        except OSError as e:
            raise MxqLibraryError(f"cannot load {library_path}: {e}") from e
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _status_name(status):
    try:
        return lib().mxq_status_string(status).decode()
    except MxqLibraryError:
        return str(status)


def _check(fn, status):
    if status != 0:
        raise MxqError(fn, status, lib().mxq_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def mxq_version():
    """Library ABI version, major*10000 + minor*100 + patch (100 = 0.1.0)."""
    return lib().mxq_version()


def mxq_arch_supported(major, minor):
    """True when the library runs on a device of this compute capability (10.3 only)."""
    return bool(lib().mxq_arch_supported(major, minor))


def mxq_inv_rope_group_quant(x, pos=None, cos=None, sin=None, R=0, q=None, sc=None,
                             err_flag=None, stream=None):
    """x bf16 [T, G, D] -> (codes uint8 [T, G, D], scales uint8 [T, G, ceil(D/128)]).

    cos/sin: bf16 [max_pos, >= R/2] (row stride = cos.stride(0)); pos int64 [T]."""
    T, G, D = x.shape
    KG = (D + 127) // 128
    if q is None:
        q = torch.empty((T, G, D), dtype=torch.uint8, device=x.device)
    if sc is None:
        sc = torch.empty((T, G, KG), dtype=torch.uint8, device=x.device)
    cs_ld = cos.stride(0) if cos is not None else 0
    max_pos = cos.shape[0] if cos is not None else 0
    st = lib().mxq_inv_rope_group_quant(_ptr(x), T, G, D, R, _ptr(pos), _ptr(cos), _ptr(sin),
                                        cs_ld, max_pos, _ptr(q), _ptr(sc), _ptr(err_flag),
                                        _stream(stream))
    _check("mxq_inv_rope_group_quant", st)
    return q, sc


def mxq_weight_scale_bytes(B, N, K):
    """Bytes of the prepared weight scales of B matrices [N, K] (0 for invalid sizes)."""
    return lib().mxq_weight_scale_bytes(B, N, K)


def mxq_prepare_weight_scales(w_e8m0, K, out=None, stream=None):
    """w_e8m0 uint8 [B, N, ceil(K/128)] -> prepared scale bytes for mxq_bmm_a8w8."""
    B, N, _ = w_e8m0.shape
    if out is None:
        out = torch.empty(mxq_weight_scale_bytes(B, N, K), dtype=torch.uint8, device=w_e8m0.device)
    st = lib().mxq_prepare_weight_scales(_ptr(w_e8m0), B, N, K, _ptr(out), _stream(stream))
    _check("mxq_prepare_weight_scales", st)
    return out


def mxq_bmm_workspace_bytes(T, G, N, K):
    """Workspace bytes of mxq_bmm_a8w8 (0 for every shape)."""
    return lib().mxq_bmm_workspace_bytes(T, G, N, K)


def mxq_bmm_a8w8(a, a_sf, w, w_sf, out=None, ws=None, stream=None):
    """a uint8 [T, G, K], a_sf uint8 [T, G, KG], w uint8 [G, N, K], w_sf prepared
    -> out bf16 [T, G, N]."""
    T, G, K = a.shape
    N = w.shape[1]
    if out is None:
        out = torch.empty((T, G, N), dtype=torch.bfloat16, device=a.device)
    need = mxq_bmm_workspace_bytes(T, G, N, K)
    if ws is None and need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device=a.device)
    st = lib().mxq_bmm_a8w8(_ptr(a), _ptr(a_sf), _ptr(w), _ptr(w_sf), _ptr(out), T, G, N, K,
                            _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))
    _check("mxq_bmm_a8w8", st)
    return out


def mxq_linear_workspace_bytes(M, N, K):
    """Workspace bytes of mxq_linear: 0 for M <= 32, else codes, scales and (M > 128) job counters."""
    return lib().mxq_linear_workspace_bytes(M, N, K)


def mxq_linear(x, w, w_sf, out=None, ws=None, stream=None):
    """x bf16 [M, K], w uint8 [N, K], w_sf prepared (B=1) -> out bf16 [M, N]
    (one launch for M <= 32 and for M > 128; quantiser + GEMM in between)."""
    M, K = x.shape
    N = w.shape[-2]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = mxq_linear_workspace_bytes(M, N, K)
    if ws is None and need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    st = lib().mxq_linear(_ptr(x), _ptr(w), _ptr(w_sf), _ptr(out), M, N, K, _ptr(ws),
                          0 if ws is None else ws.numel(), _stream(stream))
    _check("mxq_linear", st)
    return out


def mxq_linear_noalloc(x, w, w_sf, out=None, stream=None):
    """mxq_linear with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate; see include/mxq.h for the size limit and
    the rule that overlapping calls race)."""
    M, K = x.shape
    N = w.shape[-2]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    st = lib().mxq_linear_noalloc(_ptr(x), _ptr(w), _ptr(w_sf), _ptr(out), M, N, K, _stream(stream))
    _check("mxq_linear_noalloc", st)
    return out


def mxq_dequant_bf16(w, w_e8m0, out=None, stream=None):
    """w uint8 [B, N, K], w_e8m0 uint8 [B, N, ceil(K/128)] -> bf16 [B, N, K]."""
    B, N, K = w.shape
    if out is None:
        out = torch.empty((B, N, K), dtype=torch.bfloat16, device=w.device)
    st = lib().mxq_dequant_bf16(_ptr(w), _ptr(w_e8m0), _ptr(out), B, N, K, _stream(stream))
    _check("mxq_dequant_bf16", st)
    return out


def mxq_scales_f32_to_e8m0(s, out=None, err_flag=None, stream=None):
    """FP32 power-of-two scales (any shape) -> E8M0 bytes of the same shape.

    A value that is not a positive power of two in [2^-127, 2^127] gives byte
    0xFF and sets MXQ_DEVERR_SCALE in the optional int32 `err_flag`."""
    n = s.numel()
    if out is None:
        out = torch.empty(s.shape, dtype=torch.uint8, device=s.device)
    st = lib().mxq_scales_f32_to_e8m0(_ptr(s), n, _ptr(out), _ptr(err_flag), _stream(stream))
    _check("mxq_scales_f32_to_e8m0", st)
    return out


def mxq_watchdog_read(clear=False):
    """The device watchdog word (0: no bounded wait inside a kernel ever ran out)."""
    v = ctypes.c_uint32(0)
    _check("mxq_watchdog_read", lib().mxq_watchdog_read(ctypes.byref(v), 1 if clear else 0))
    return v.value


def mxq_debug_set_pair_limit(pairs):
    """Testing aid: cap the CTA pairs of the many-token GEMM launches (0 = no
    cap); returns the previous cap."""
    return lib().mxq_debug_set_pair_limit(int(pairs))


def mxq_debug_set_lazy_pairs(first):
    """Testing aid: pairs of the one-launch prefill from index `first` on skip
    their quantisation jobs (negative: none); returns the previous setting."""
    return lib().mxq_debug_set_lazy_pairs(int(first))


def mxq_debug_takeovers(clear=False):
    """Testing aid: prefill quantisation jobs quantised by a waiting pair
    instead of their owner since the last clear."""
    v = ctypes.c_uint32(0)
    _check("mxq_debug_takeovers", lib().mxq_debug_takeovers(ctypes.byref(v), 1 if clear else 0))
    return v.value


def mxq_watchdog_selftest(limit_ns=1_000_000, stream=None):
    """Launch a kernel whose only wait never completes; it gives up after
    `limit_ns` and sets the watchdog word (no fault, the context stays usable)."""
    _check("mxq_watchdog_selftest", lib().mxq_watchdog_selftest(limit_ns, _stream(stream)))


def mxq_wo_a_workspace_bytes(T, G, D, N):
    """Workspace bytes of mxq_wo_a: 0 for T <= 32, else codes, scales and (T > 128) job counters."""
    return lib().mxq_wo_a_workspace_bytes(T, G, D, N)


def mxq_wo_a(x, pos, cos, sin, w, w_sf, R=64, out=None, ws=None, err_flag=None, stream=None):
    """The wo_a projection in one library call: x bf16 [T, G, D] -> out bf16 [T, G, N]
    (one launch for T <= 32 and for T > 128, where the GEMM quantises x itself;
    quantiser + GEMM in between).  `ws` (mxq_wo_a_workspace_bytes) is allocated
    when not given; concurrent calls need distinct workspaces."""
    T, G, D = x.shape
    N = w.shape[1]
    if out is None:
        out = torch.empty((T, G, N), dtype=torch.bfloat16, device=x.device)
    need = mxq_wo_a_workspace_bytes(T, G, D, N)
    if ws is None and need > 0:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    cs_ld = cos.stride(0) if cos is not None else 0
    max_pos = cos.shape[0] if cos is not None else 0
    st = lib().mxq_wo_a(_ptr(x), _ptr(pos), _ptr(cos), _ptr(sin), cs_ld, max_pos, _ptr(w), _ptr(w_sf),
                        _ptr(out), T, G, D, N, R, _ptr(err_flag), _ptr(ws),
                        0 if ws is None else ws.numel(), _stream(stream))
    _check("mxq_wo_a", st)
    return out


wo_a = mxq_wo_a


def mxq_rope_kv_insert(q, kv, pos, cos, sin, R, slot_mapping, cache, scale=None, q_out=None,
                       err_flag=None, stream=None):
    """Forward RoPE of q bf16 [T, H, Dq] (into q_out, default a new tensor;
    pass q_out=q to rotate in place) and of kv bf16 [T, Dk], whose rows are
    written to cache[slot_mapping[t]]: uint8 cache [num_slots, Dk] = E4M3 of
    fl32(y / scale) with `scale` a float32 device tensor of one element, or
    bf16 cache [num_slots, Dk] = bf16(y).  Returns q_out."""
    T, H, Dq = q.shape if q is not None else (kv.shape[0], 0, 0)
    Dk = kv.shape[1]
    if q is not None and q_out is None:
        q_out = torch.empty_like(q)
    if cache.dtype == torch.uint8:
        dtype = MXQ_CACHE_E4M3
    elif cache.dtype == torch.bfloat16:
        dtype = MXQ_CACHE_BF16
    else:
        raise MxqError("mxq_rope_kv_insert", 4, "cache must be uint8 (E4M3) or bfloat16")
    cs_ld = cos.stride(0) if cos is not None else 0
    max_pos = cos.shape[0] if cos is not None else 0
    st = lib().mxq_rope_kv_insert(_ptr(q), _ptr(q_out), T, H, Dq, _ptr(kv), Dk, _ptr(pos), _ptr(cos),
                                  _ptr(sin), cs_ld, max_pos, R, _ptr(slot_mapping), _ptr(cache),
                                  cache.shape[0], dtype, _ptr(scale), _ptr(err_flag), _stream(stream))
    _check("mxq_rope_kv_insert", st)
    return q_out
