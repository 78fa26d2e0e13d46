"""fa_decode_noalloc: split-KV decode for callers that cannot allocate.

Some callers cannot call cudaMalloc or hand the library a workspace -- a
plugin inside a host framework that owns all device memory, or a
latency-critical loop where an allocation could stall the device.  For them
fa_decode_noalloc keeps its split partials in a fixed scratch array inside
the library.  These tests call it through the C ABI and check it

* against the fp64 oracle at the decode tolerances the other GPU tests use
  (O max 2e-2, mean 2e-3; LSE 1e-3), and
* against the ordinary entry point fa_decode_ex (which takes a workspace)
  bit for bit: both launch the same two kernels with the same split, so
  any difference would mean a partial was read from the wrong place,

on two calls in a row, with and without an LSE output, and on a call that
fills the whole scratch followed by a small one (so the leftovers of the
first sit next to the parts the second reads).  A request larger than the
scratch is refused.  The file is named so that pytest collects it last.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3
MAX_PARTS = 16384          # B * H * num_splits the scratch holds


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _with_workspace(q, kc, vc, splits, scale, want_lse=True):
    B, H, L, d = kc.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H), device="cuda", dtype=torch.float32) if want_lse else None
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_DECODE, B, H, L, d, splits),
                     dtype=torch.uint8, device="cuda")
    _lib.check(_lib.fa_decode_ex(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                 lse.data_ptr() if want_lse else None, B, H, L, d, splits, scale,
                                 ws.data_ptr(), ws.numel(), _stream()))
    return o, lse


def _noalloc(q, kc, vc, splits, scale, want_lse=True):
    B, H, L, d = kc.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H), device="cuda", dtype=torch.float32) if want_lse else None
    _lib.check(_lib.fa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                      lse.data_ptr() if want_lse else None, B, H, L, d, splits,
                                      scale, _stream()))
    return o, lse


def _check(q, kc, vc, splits, want_lse=True):
    scale = 1 / math.sqrt(q.shape[-1])
    o, lse = _noalloc(q, kc, vc, splits, scale, want_lse)
    assert _lib.fa_get_device_status(_stream()) == 0, _lib.fa_last_error()
    o_ex, lse_ex = _with_workspace(q, kc, vc, splits, scale, want_lse)
    assert torch.equal(o, o_ex)
    if want_lse:
        assert torch.equal(lse, lse_ex)
    o_ref, lse_ref = orc.attention_decode(_f64(q), _f64(kc), _f64(vc), scale)
    err = np.abs(_f64(o) - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    if want_lse:
        assert np.abs(_f64(lse) - lse_ref).max() <= LSE_MAX


def test_noalloc_two_calls_in_a_row():
    # Two different problems back to back: the second call must not see
    # anything the first one left in the shared scratch.
    for B, H, L, splits, seed in [(4, 8, 3000, 7, 11), (2, 16, 1025, 16, 12)]:
        q, kc, vc = inputs.decode_inputs(B, H, L, 128, torch.bfloat16, seed, "cuda")
        _check(q, kc, vc, splits)


def test_noalloc_without_lse_output():
    q, kc, vc = inputs.decode_inputs(3, 4, 2049, 128, torch.bfloat16, 14, "cuda")
    _check(q, kc, vc, 5, want_lse=False)
    _check(q, kc, vc, 5, want_lse=True)


def test_noalloc_full_scratch_then_small_call():
    # 8 * 32 * 64 = 16384 parts: every slot of the scratch written; then a
    # call with 2 * 3 * 3 = 18 parts whose partials sit among the leftovers.
    q, kc, vc = inputs.decode_inputs(8, 32, 4096, 128, torch.bfloat16, 15, "cuda")
    assert 8 * 32 * 64 == MAX_PARTS
    _check(q, kc, vc, 64)
    q, kc, vc = inputs.decode_inputs(2, 3, 700, 128, torch.bfloat16, 16, "cuda")
    _check(q, kc, vc, 3)
    _check(q, kc, vc, 3, want_lse=False)


def test_noalloc_rejects_requests_beyond_the_scratch():
    q, kc, vc = inputs.decode_inputs(1, 2, 64, 128, torch.bfloat16, 13, "cuda")
    o = torch.empty_like(q)
    # B * H * num_splits = 64 * 32 * 16 = 32768 > 16384 parts: refused before
    # any launch (the pointers are never dereferenced).
    code = _lib.fa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None,
                                  64, 32, 64, 128, 16, 0.1, _stream())
    assert code == _lib.FA_ERR_UNSUPPORTED
    assert "scratch" in _lib.fa_last_error()
