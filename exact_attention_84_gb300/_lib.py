"""ctypes binding of libfa.so: the C-ABI entry points under the same names.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these symbols.  Pointers are passed as Python ints (device
addresses), streams as ``cudaStream_t`` handles (ints).  If the shared
library has not been built, loading fails loudly; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_NO_MEMORY = 5
FA_OP_FORWARD, FA_OP_BACKWARD, FA_OP_DECODE, FA_OP_FORWARD_FP8 = 0, 1, 2, 3

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

# name -> (restype, argtypes), mirroring include/fa.h
SIGNATURES = {
    "fa_forward": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_forward_fp32": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_forward_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P]),
    "fa_forward_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _F, _F, _I, _I,
                            _P, _P, _Z, _P]),
    "fa_backward_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I,
                             _I, _P, _I, _P, _Z, _P]),
    "fa_decode_gqa": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _Z, _P]),
    "fa_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_backward_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I,
                            _P, _Z, _P]),
    "fa_decode": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "fa_decode_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _Z, _P]),
    "fa_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "fa_decode_splits": (_I, [_I, _I, _I, _I]),
    "fa_get_device_status": (_I, [_P]),
    "fa_set_timing_events": (_I, [_P, _P]),
    "fa_selftest_timeout": (_I, [ctypes.c_uint, _P]),
    "fa_last_error": (ctypes.c_char_p, []),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libfa error {code}: {msg}")
        self.code = code


def load() -> ctypes.CDLL:
    """Load libfa.so (built in-tree by ``exact_attention_84_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m exact_attention_84_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _call(name, *args):
    return getattr(load(), name)(*args)


def check(code: int) -> None:
    """Raise FAError for a non-zero status, with the library's message."""
    if code != FA_OK:
        raise FAError(code, fa_last_error())


def fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal, stream):
    return _call("fa_forward", q, k, v, o, lse, B, H, N, d, scale, causal, stream)


def fa_forward_fp32(q, k, v, o, lse, B, H, N, d, scale, causal, stream):
    return _call("fa_forward_fp32", q, k, v, o, lse, B, H, N, d, scale, causal, stream)


def fa_forward_gqa(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, window, alibi_slopes,
                   stream):
    return _call("fa_forward_gqa", q, k, v, o, lse, B, Hq, Hkv, N, d, scale, causal, window,
                 alibi_slopes, stream)


def fa_forward_fp8(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, q_descale, k_descale, v_descale,
                   causal, window, alibi_slopes, ws, ws_bytes, stream):
    return _call("fa_forward_fp8", q, k, v, o, lse, B, Hq, Hkv, N, d, scale, q_descale,
                 k_descale, v_descale, causal, window, alibi_slopes, ws, ws_bytes, stream)


def fa_backward_gqa(q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, scale, causal, window,
                    alibi_slopes, deterministic, ws, ws_bytes, stream):
    return _call("fa_backward_gqa", q, k, v, o, lse, dO, dq, dk, dv, B, Hq, Hkv, N, d, scale,
                 causal, window, alibi_slopes, deterministic, ws, ws_bytes, stream)


def fa_decode_gqa(q, kcache, vcache, o, lse_out, B, Hq, Hkv, Lkv, d, num_splits, scale,
                  alibi_slopes, ws, ws_bytes, stream):
    return _call("fa_decode_gqa", q, kcache, vcache, o, lse_out, B, Hq, Hkv, Lkv, d, num_splits,
                 scale, alibi_slopes, ws, ws_bytes, stream)


def fa_backward(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, stream):
    return _call("fa_backward", q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal,
                 stream)


def fa_backward_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes,
                   stream):
    return _call("fa_backward_ex", q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal,
                 ws, ws_bytes, stream)


def fa_decode(q, kcache, vcache, o, B, H, Lkv, d, num_splits, stream):
    return _call("fa_decode", q, kcache, vcache, o, B, H, Lkv, d, num_splits, stream)


def fa_decode_ex(q, kcache, vcache, o, lse_out, B, H, Lkv, d, num_splits, scale, ws, ws_bytes,
                 stream):
    return _call("fa_decode_ex", q, kcache, vcache, o, lse_out, B, H, Lkv, d, num_splits, scale,
                 ws, ws_bytes, stream)


def fa_decode_noalloc(q, kcache, vcache, o, lse_out, B, H, Lkv, d, num_splits, scale, stream):
    return _call("fa_decode_noalloc", q, kcache, vcache, o, lse_out, B, H, Lkv, d, num_splits,
                 scale, stream)


def fa_decode_splits(B, Hq, Hkv, Lkv):
    return _call("fa_decode_splits", B, Hq, Hkv, Lkv)


def fa_workspace_size(op, B, H, n_or_lkv, d, num_splits):
    return _call("fa_workspace_size", op, B, H, n_or_lkv, d, num_splits)


def fa_get_device_status(stream):
    return _call("fa_get_device_status", stream)


def fa_selftest_timeout(limit_ms, stream):
    return _call("fa_selftest_timeout", limit_ms, stream)


def fa_set_timing_events(before, after):
    return _call("fa_set_timing_events", before, after)


def fa_last_error() -> str:
    msg = _call("fa_last_error")
    return msg.decode() if msg else ""
