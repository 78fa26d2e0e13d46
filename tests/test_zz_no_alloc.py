"""fa_decode_noalloc: split-KV decode for callers that cannot allocate.

Some callers cannot call cudaMalloc or hand the library a workspace -- a
plugin inside a host framework that owns all device memory, or a
latency-critical loop where an allocation could stall the device.  For them
fa_decode_noalloc keeps its split partials in a fixed scratch array inside
the library.  These tests call it through the C ABI and check it against the
ordinary entry point (fa_decode_ex, which takes a workspace) on two calls in
a row, at the decode tolerances the other GPU tests use, and check that a
request larger than the scratch is refused.  The file is named so that pytest
collects it last.
"""

import math

import numpy as np
import pytest
import torch

from exact_attention_84_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _reference(q, kc, vc, splits, scale):
    B, H, L, d = kc.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H), device="cuda", dtype=torch.float32)
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_DECODE, B, H, L, d, splits),
                     dtype=torch.uint8, device="cuda")
    _lib.check(_lib.fa_decode_ex(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, H, L, d, splits, scale, ws.data_ptr(),
                                 ws.numel(), _stream()))
    return o, lse


def _noalloc(q, kc, vc, splits, scale):
    B, H, L, d = kc.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H), device="cuda", dtype=torch.float32)
    _lib.check(_lib.fa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), B, H, L, d, splits, scale, _stream()))
    return o, lse


def test_noalloc_matches_decode_ex_on_two_calls_in_a_row():
    scale = 1 / math.sqrt(128)
    # Two different problems back to back: the second call must not see
    # anything the first one left in the shared scratch.
    cases = [(4, 8, 3000, 7, 11), (2, 16, 1025, 16, 12)]
    for B, H, L, splits, seed in cases:
        q, kc, vc = inputs.decode_inputs(B, H, L, 128, torch.bfloat16, seed, "cuda")
        o_ref, lse_ref = _reference(q, kc, vc, splits, scale)
        o, lse = _noalloc(q, kc, vc, splits, scale)
        assert _lib.fa_get_device_status(_stream()) == 0, _lib.fa_last_error()
        d = (o.float() - o_ref.float()).abs()
        assert d.max().item() <= O_MAX and d.mean().item() <= O_MEAN
        assert (lse - lse_ref).abs().max().item() <= LSE_MAX
        assert np.isfinite(o.float().cpu().numpy()).all()


def test_noalloc_rejects_requests_beyond_the_scratch():
    q, kc, vc = inputs.decode_inputs(1, 2, 64, 128, torch.bfloat16, 13, "cuda")
    o = torch.empty_like(q)
    # B * H * num_splits = 64 * 32 * 16 = 32768 > 16384 parts: refused before
    # any launch (the pointers are never dereferenced).
    code = _lib.fa_decode_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None,
                                  64, 32, 64, 128, 16, 0.1, _stream())
    assert code == _lib.FA_ERR_UNSUPPORTED
    assert "scratch" in _lib.fa_last_error()
