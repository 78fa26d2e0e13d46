"""Torch-facing convenience layer over the C-ABI.

PyTorch only owns device memory and streams here: each function allocates
its outputs with ``torch.empty`` and hands raw pointers to one C-ABI call on
the current CUDA stream.  Inputs must be contiguous CUDA tensors of the
documented dtype; nothing is converted or computed on the Python side.
"""

from __future__ import annotations

import math

import torch

from . import _lib


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need(t: torch.Tensor, dtype: torch.dtype, name: str):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def _slopes(alibi_slopes, heads):
    if alibi_slopes is None:
        return None
    _need(alibi_slopes, torch.float32, "alibi_slopes")
    if alibi_slopes.numel() != heads:
        raise ValueError(f"alibi_slopes needs {heads} entries")
    return alibi_slopes.data_ptr()


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            window: int = 0, alibi_slopes=None):
    """O, LSE = attention(q, k, v) for [B, H, N, d] bf16 (or fp32) tensors.

    bf16 only: k and v may have fewer heads Hkv (H a multiple of Hkv; query
    head h reads key/value head h // (H // Hkv)), ``window`` w >= 1 (with
    ``causal``) lets query i see keys i-w+1 .. i only, and ``alibi_slopes``
    (a CUDA fp32 tensor of H slopes) adds -slope_h * |i - j| to the scores."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    fp32 = q.dtype == torch.float32
    dtype = torch.float32 if fp32 else torch.bfloat16
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, dtype, n)
    o = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32) if lse is None else lse
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr())
    if Hkv != H or window or alibi_slopes is not None:
        if fp32:
            raise ValueError("grouped heads, windows and ALiBi need bf16 tensors")
        _lib.check(_lib.fa_forward_gqa(*ptrs, B, H, Hkv, N, d, scale, int(causal), int(window),
                                       _slopes(alibi_slopes, H), _stream()))
    else:
        fn = _lib.fa_forward_fp32 if fp32 else _lib.fa_forward
        _lib.check(fn(*ptrs, B, H, N, d, scale, int(causal), _stream()))
    return o, lse


def forward_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                causal: bool = False, scale: float | None = None, window: int = 0, out=None,
                lse=None, workspace=None, alibi_slopes=None):
    """O (bf16), LSE for E4M3 inputs held as uint8 codes: q8 [B, H, N, d],
    k8, v8 [B, Hkv, N, d]; real values are code * descale."""
    B, H, N, d = q8.shape
    Hkv = k8.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _need(t, torch.uint8, n)
    o = torch.empty(q8.shape, device=q8.device, dtype=torch.bfloat16) if out is None else out
    lse = torch.empty((B, H, N), device=q8.device, dtype=torch.float32) if lse is None else lse
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _lib.check(_lib.fa_forward_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, Hkv, N, d, scale, q_descale, k_descale,
                                   v_descale, int(causal), int(window),
                                   _slopes(alibi_slopes, H), ws_ptr, ws_bytes, _stream()))
    return o, lse


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
             workspace=None, out=None, window: int = 0, alibi_slopes=None,
             deterministic: bool = False):
    """dQ, dK, dV for bf16 [B, H, N, d] tensors; lse from ``forward``.
    ``out`` may hold three preallocated tensors (dq, dk, dv) to write into.
    k, v (and dk, dv) may have fewer heads, and ``window`` / ``alibi_slopes``
    apply, as in ``forward``.  ``deterministic``: bitwise-reproducible dQ
    (no atomics)."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
        for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
            _need(t, torch.bfloat16, n)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    args = ptrs + (B, H, N, d, scale, int(causal))
    if Hkv != H or window or alibi_slopes is not None or deterministic:
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _lib.check(_lib.fa_backward_gqa(*ptrs, B, H, Hkv, N, d, scale, int(causal), int(window),
                                        _slopes(alibi_slopes, H), int(deterministic), ws_ptr,
                                        ws_bytes, _stream()))
    elif workspace is None:
        _lib.check(_lib.fa_backward(*args, _stream()))
    else:
        _lib.check(_lib.fa_backward_ex(*args, workspace.data_ptr(), workspace.numel() *
                                       workspace.element_size(), _stream()))
    return dq, dk, dv


def decode(q, kcache, vcache, num_splits: int = 1, scale: float | None = None,
           with_lse: bool = False, workspace=None, alibi_slopes=None):
    """o (and optionally lse) for one query token per (b, h): q [B, H, d],
    caches [B, Hkv, Lkv, d], all bf16 (H a multiple of Hkv: query head h
    reads cache head h // (H // Hkv)).  ``alibi_slopes``: H fp32 slopes; the
    new token is at position Lkv - 1.  ``num_splits=0`` lets the library
    choose (grouped or ALiBi calls)."""
    B, Hkv, L, d = kcache.shape
    H = q.shape[1]
    for t, n in ((q, "q"), (kcache, "kcache"), (vcache, "vcache")):
        _need(t, torch.bfloat16, n)
    o = torch.empty_like(q)
    lse = torch.empty((B, H), device=q.device, dtype=torch.float32) if with_lse else None
    if Hkv != H or alibi_slopes is not None or num_splits == 0:
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _lib.check(_lib.fa_decode_gqa(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                      o.data_ptr(), lse.data_ptr() if lse is not None else None,
                                      B, H, Hkv, L, d, num_splits, scale,
                                      _slopes(alibi_slopes, H), ws_ptr, ws_bytes, _stream()))
    elif scale is None and not with_lse and workspace is None:
        _lib.check(_lib.fa_decode(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                  o.data_ptr(), B, H, L, d, num_splits, _stream()))
    else:
        scale = 1.0 / math.sqrt(d) if scale is None else scale
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _lib.check(_lib.fa_decode_ex(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                     o.data_ptr(), lse.data_ptr() if lse is not None else None,
                                     B, H, L, d, num_splits, scale, ws_ptr, ws_bytes,
                                     _stream()))
    return (o, lse) if with_lse else o


def device_status() -> int:
    """Synchronise the current stream and return the kernels' status word."""
    return _lib.fa_get_device_status(_stream())


class _Attention(torch.autograd.Function):
    """Autograd node over ``forward`` / ``backward`` (bf16): saves Q, K, V,
    O and LSE, and returns dQ, dK, dV from the recomputation backward."""

    @staticmethod
    def forward(ctx, q, k, v, causal, scale, window, alibi_slopes, deterministic):
        o, lse = forward(q, k, v, causal=causal, scale=scale, window=window,
                         alibi_slopes=alibi_slopes)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.opts = (causal, scale, window, alibi_slopes, deterministic)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        causal, scale, window, alibi_slopes, deterministic = ctx.opts
        dq, dk, dv = backward(q, k, v, o, lse, do.contiguous(), causal=causal, scale=scale,
                              window=window, alibi_slopes=alibi_slopes,
                              deterministic=deterministic)
        return dq, dk, dv, None, None, None, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None, window: int = 0,
              alibi_slopes=None, deterministic: bool = False):
    """Differentiable attention for bf16 [B, H, N, d] q and [B, Hkv, N, d]
    k, v: O = softmax(scale Q K^T [+ mask, ALiBi]) V, with dQ, dK, dV from
    the library's backward when autograd asks for them."""
    return _Attention.apply(q, k, v, causal, scale, window, alibi_slopes, deterministic)
