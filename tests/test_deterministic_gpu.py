"""Deterministic backward (dQ by query blocks in a fixed key order, no
atomics): parity with the oracle at the backward tolerance (5e-2), and
bitwise-identical gradients from run to run."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import api, inputs
from gpu_common import G_MAX, guarded, guards_intact, np64, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu

D = 128
SCALE = 1 / math.sqrt(D)


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 1, 1, 1), (1, 2, 2, 64), (2, 2, 1, 200),
                                        (1, 4, 2, 300), (1, 1, 1, 520)])
@pytest.mark.parametrize("causal,window,alibi", [(False, 0, False), (True, 0, False),
                                                 (True, 90, False), (True, 0, True)])
def test_deterministic_backward(B, Hq, Hkv, N, causal, window, alibi):
    q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 120 + N, "cuda",
                                    with_do=True)
    slopes = inputs.alibi_slopes(Hq, "cuda") if alibi else None
    o, lse = api.forward(q, k, v, causal=causal, scale=SCALE, window=window, alibi_slopes=slopes)
    bq, dq = guarded((B, Hq, N, D), torch.bfloat16)
    bk, dk = guarded((B, Hkv, N, D), torch.bfloat16)
    bv, dv = guarded((B, Hkv, N, D), torch.bfloat16)
    api.backward(q, k, v, o, lse, do, causal=causal, scale=SCALE, window=window,
                 alibi_slopes=slopes, deterministic=True, out=(dq, dk, dv))
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), SCALE, causal,
                                      window or None, np64(slopes) if alibi else None)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(np64(got) - ref).max()
        assert err <= G_MAX, f"{name} max err {err:.3e} (N={N} causal={causal} w={window})"
    assert guards_intact(bq) and guards_intact(bk) and guards_intact(bv)
    # a second run gives the same bits
    g2 = api.backward(q, k, v, o, lse, do, causal=causal, scale=SCALE, window=window,
                      alibi_slopes=slopes, deterministic=True)
    for a, b in zip((dq, dk, dv), g2):
        assert torch.equal(a, b)


def test_deterministic_train_b8_h32_n4096():
    """The training workload: bitwise-equal gradients over three runs,
    agreement with the atomic dQ within the tolerance, and sampled heads
    against the oracle."""
    w = inputs.TRAIN_N4096
    q, k, v, do = inputs.workload_inputs(w, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE)
    runs = [api.backward(q, k, v, o, lse, do, causal=True, scale=SCALE, deterministic=True)
            for _ in range(3)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a, b)
    atomic = api.backward(q, k, v, o, lse, do, causal=True, scale=SCALE)
    assert torch.equal(atomic[1], runs[0][1]) and torch.equal(atomic[2], runs[0][2])
    assert (atomic[0].float() - runs[0][0].float()).abs().max().item() <= G_MAX
    dq, dk, dv = runs[0]
    for b, h in ((0, 0), (7, 31)):
        qh, kh, vh, doh = (np64(t[b, h]) for t in (q, k, v, do))
        refs = orc.attention_backward(qh[None], kh[None], vh[None], doh[None], SCALE, True)
        for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
            err = np.abs(np64(got[b, h]) - ref[0]).max()
            assert err <= G_MAX, f"{name} ({b},{h}) max err {err:.3e}"
