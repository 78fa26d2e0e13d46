"""Grouped query heads and the causal sliding window against the oracle:
forward (O, LSE), backward (dQ, dK, dV summed over each group) and split-KV
decode.  Same tolerances as the per-head paths (max 2e-2 / mean 2e-3 on O,
1e-3 on LSE, 5e-2 on gradients)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import (G_MAX, O_MAX, assert_close_bf16, guarded, guards_intact, np64,
                        status_clean)  # noqa: F401

pytestmark = pytest.mark.gpu

D = 128
SCALE = 1 / math.sqrt(D)

# (B, Hq, Hkv, N): groups of 1, 2, 3, 4 and 8; several tiles and ragged tails
FWD_SHAPES = [(1, 4, 1, 300), (2, 6, 2, 257), (1, 3, 3, 129), (1, 8, 2, 640), (1, 2, 1, 1)]
# (causal, window)
MASKS = [(False, 0), (True, 0), (True, 1), (True, 100), (True, 128), (True, 200),
         (True, 5000)]


@pytest.mark.parametrize("B,Hq,Hkv,N", FWD_SHAPES)
@pytest.mark.parametrize("causal,window", MASKS)
def test_forward_gqa_window(B, Hq, Hkv, N, causal, window):
    q, k, v = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 50 + N + Hq, "cuda")
    bo, o = guarded((B, Hq, N, D), torch.bfloat16)
    bl, lse = guarded((B, Hq, N), torch.float32)
    api.forward(q, k, v, causal=causal, scale=SCALE, out=o, lse=lse, window=window)
    o_ref, lse_ref = orc.attention_forward_gqa(np64(q), np64(k), np64(v), SCALE, causal,
                                               window or None)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"N={N} g={Hq // Hkv} w={window}")
    assert guards_intact(bo) and guards_intact(bl)


def test_forward_window_one_is_v():
    """Width 1: each query sees only its own key, so O = V and LSE is that
    one scaled score."""
    q, k, v = inputs.gqa_inputs(1, 4, 2, 333, D, torch.bfloat16, 9, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE, window=1)
    vr = v.repeat_interleave(2, dim=1)
    assert (o.float() - vr.float()).abs().max().item() <= 1e-2
    ref = (q.float() * k.repeat_interleave(2, dim=1).float()).sum(-1) * SCALE
    assert (lse - ref).abs().max().item() <= 1e-3


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 1, 200), (2, 4, 2, 256), (1, 6, 2, 130),
                                        (1, 2, 2, 520), (1, 8, 1, 64)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 1), (True, 70),
                                           (True, 300)])
def test_backward_gqa_window(B, Hq, Hkv, N, causal, window):
    q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 60 + N, "cuda",
                                    with_do=True)
    o, lse = api.forward(q, k, v, causal=causal, scale=SCALE, window=window)
    bq, dq = guarded((B, Hq, N, D), torch.bfloat16)
    bk, dk = guarded((B, Hkv, N, D), torch.bfloat16)
    bv, dv = guarded((B, Hkv, N, D), torch.bfloat16)
    api.backward(q, k, v, o, lse, do, causal=causal, scale=SCALE, out=(dq, dk, dv),
                 window=window)
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), SCALE, causal,
                                      window or None)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(np64(got) - ref).max()
        assert err <= G_MAX, f"{name} max err {err:.3e} (N={N} g={Hq // Hkv} w={window})"
    assert guards_intact(bq) and guards_intact(bk) and guards_intact(bv)


def test_backward_gqa_caller_workspace():
    B, Hq, Hkv, N = 1, 4, 2, 300
    q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 3, "cuda", with_do=True)
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE, window=90)
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_BACKWARD, B, Hq, N, D, 0),
                     dtype=torch.uint8, device="cuda")
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True, scale=SCALE, workspace=ws,
                              window=90)
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), SCALE, True, 90)
    for got, ref in zip((dq, dk, dv), refs):
        assert np.abs(np64(got) - ref).max() <= G_MAX


@pytest.mark.parametrize("B,Hq,Hkv,L,splits", [
    (B, Hq, Hkv, L, s)
    for (B, Hq, Hkv, L) in [(1, 4, 1, 1), (2, 8, 2, 1000), (1, 32, 1, 513), (3, 12, 4, 64),
                            (1, 20, 1, 100), (2, 8, 8, 300)]
    for s in [1, 3, 8] if s <= L])
def test_decode_gqa(B, Hq, Hkv, L, splits):
    q, kc, vc = inputs.decode_gqa_inputs(B, Hq, Hkv, L, D, torch.bfloat16, 70 + L, "cuda")
    bo, o_view = guarded((B, Hq, D), torch.bfloat16)
    o, lse = api.decode(q, kc, vc, num_splits=splits, scale=SCALE, with_lse=True)
    o_ref, lse_ref = orc.attention_decode_gqa(np64(q), np64(kc), np64(vc), SCALE)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"L={L} g={Hq // Hkv} splits={splits}")
    # through the C-ABI into a guarded output and a caller workspace
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_DECODE, B, Hq, L, D, splits),
                     dtype=torch.uint8, device="cuda")
    _lib.check(_lib.fa_decode_gqa(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o_view.data_ptr(),
                                  None, B, Hq, Hkv, L, D, splits, SCALE, None, ws.data_ptr(),
                                  ws.numel(), torch.cuda.current_stream().cuda_stream))
    assert torch.equal(o_view, o)
    assert guards_intact(bo)


# ------------------------------------------------------- automatic split count
@pytest.mark.parametrize("B,Hq,Hkv,L", [(2, 8, 2, 5000), (4, 4, 4, 3000)])
def test_decode_automatic_splits(B, Hq, Hkv, L):
    q, kc, vc = inputs.decode_gqa_inputs(B, Hq, Hkv, L, D, torch.bfloat16, 140 + L, "cuda")
    assert _lib.fa_decode_splits(B, Hq, Hkv, L) >= 1
    o, lse = api.decode(q, kc, vc, num_splits=0, scale=SCALE, with_lse=True)
    o_ref, lse_ref = orc.attention_decode_gqa(np64(q), np64(kc), np64(vc), SCALE)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"L={L} automatic splits")
