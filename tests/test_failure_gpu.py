"""Failure detection without a GPU fault: a bounded wait that runs out is
reported through fa_get_device_status and leaves the context usable, and an
injected allocation failure is reported as FA_ERR_NO_MEMORY before anything
is launched."""
import math
import os

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import assert_close_bf16, np64, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu


def _small_forward_ok():
    q, k, v = inputs.attention_inputs(1, 2, 200, 128, torch.bfloat16, 3, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=1 / math.sqrt(128))
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), 1 / math.sqrt(128), True)
    assert_close_bf16(o, lse, o_ref, lse_ref)


def test_wait_timeout_is_reported_and_context_survives():
    stream = torch.cuda.current_stream().cuda_stream
    assert api.device_status() == _lib.FA_OK
    _lib.check(_lib.fa_selftest_timeout(50, stream))
    assert api.device_status() == _lib.FA_ERR_TIMEOUT
    assert "time" in _lib.fa_last_error()
    assert api.device_status() == _lib.FA_OK          # read once, then cleared
    _small_forward_ok()                                # the context is still usable


def test_injected_allocation_failure(monkeypatch):
    B, H, N, d = 1, 2, 130, 128
    q, k, v, do = inputs.attention_inputs(B, H, N, d, torch.bfloat16, 4, "cuda", with_do=True)
    o, lse = api.forward(q, k, v, causal=True)
    dq = torch.full_like(q, 7.0)
    dk, dv = torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    monkeypatch.setenv("FA_DEBUG_FAIL_ALLOC", "1")
    with pytest.raises(_lib.FAError) as exc:
        api.backward(q, k, v, o, lse, do, causal=True, out=(dq, dk, dv))
    assert exc.value.code == _lib.FA_ERR_NO_MEMORY
    torch.cuda.synchronize()
    assert bool((dq == 7.0).all() and (dk == 7.0).all() and (dv == 7.0).all())   # nothing ran
    qd, kc, vc = inputs.decode_inputs(1, 2, 100, d, torch.bfloat16, 5, "cuda")
    with pytest.raises(_lib.FAError) as exc:
        api.decode(qd, kc, vc, num_splits=2)
    assert exc.value.code == _lib.FA_ERR_NO_MEMORY
    monkeypatch.delenv("FA_DEBUG_FAIL_ALLOC")
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True)
    refs = orc.attention_backward(np64(q), np64(k), np64(v), np64(do), 1 / math.sqrt(d), True)
    for got, ref in zip((dq, dk, dv), refs):
        assert np.abs(np64(got) - ref).max() <= 5e-2
