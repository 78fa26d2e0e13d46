"""The full-size workloads compared in full against the fp64 oracle.

Lensa ML "FlashAttention", step 6: the tiled result equals standard
attention up to rounding, so every output element of every workload is held
to the bf16 tolerances (O max 2e-2 and mean 2e-3 per head, LSE 1e-3,
gradients 5e-2), in the launch configuration the bench times:

* bf16 causal forward B1 H32 N8192: every row of every head, including head
  31 whose keys are all equal (there O is also checked against the prefix
  means of V);
* bf16 causal forward+backward B8 H32 N4096: O, LSE, dQ, dK and dV of all
  256 heads;
* split-KV decode B64 H32 Lkv32768: every (batch, head) for 1, 2, 4, 8 and
  16 splits;
* grouped-query decode B64 Hq32 Hkv8 Lkv32768: every (batch, query head) for
  1, 2, 4 and 8 splits;
* causal sliding-window (w = 1024) forward B1 H32 N8192: every row of every
  head;
* grouped-query causal forward+backward B8 Hq32 Hkv8 N4096: O, LSE, dQ, dK
  and dV of all 64 (batch, key/value head) groups, 256 query heads.

Host copies are taken once per tensor (fp32 on the host, widened to fp64
head by head inside the oracle).
"""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import api, inputs
from gpu_common import G_MAX, O_MAX, assert_close_bf16, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu


def host(t):
    return t.detach().float().cpu().numpy()


def f64(a):
    return np.asarray(a, dtype=np.float64)


def test_long_causal_n8192_every_element():
    w = inputs.LONG_CAUSAL
    q, k, v = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    o, lse = api.forward(q, k, v, causal=True, scale=scale)
    Q, K, V, O, LSE = (host(t) for t in (q, k, v, o, lse))
    for h in range(w.H):
        o_ref, lse_ref = orc.attention_forward(Q[0, h], K[0, h], V[0, h], scale, True)
        assert_close_bf16(O[0, h], LSE[0, h], o_ref, lse_ref, f"head {h}")
    # the identical-keys head: every visible key carries the same weight
    h = w.uniform_head
    mean_prefix = np.cumsum(f64(V[0, h]), axis=0) / np.arange(1, w.N + 1)[:, None]
    assert np.abs(f64(O[0, h]) - mean_prefix).max() <= O_MAX


def test_train_b8_h32_n4096_every_head():
    w = inputs.TRAIN_N4096
    q, k, v, do = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    o, lse = api.forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    Q, K, V, DO, O, LSE, DQ, DK, DV = (host(t) for t in (q, k, v, do, o, lse, dq, dk, dv))
    worst = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    for b in range(w.B):
        for h in range(w.H):
            qh, kh, vh, doh = (f64(t[b, h]) for t in (Q, K, V, DO))
            o_ref, lse_ref = orc.attention_forward(qh, kh, vh, scale, True)
            assert_close_bf16(O[b, h], LSE[b, h], o_ref, lse_ref, f"fwd ({b},{h})")
            refs = orc.attention_backward(qh[None], kh[None], vh[None], doh[None], scale, True)
            for name, got, ref in zip(("dq", "dk", "dv"), (DQ, DK, DV), refs):
                err = float(np.abs(f64(got[b, h]) - ref[0]).max())
                worst[name] = max(worst[name], err)
                assert err <= G_MAX, f"{name} ({b},{h}) max err {err:.3e}"
    print("worst gradient errors over all 256 heads:", worst)


def test_decode_b64_h32_l32768_every_head():
    w = inputs.DECODE_L32K
    q, kc, vc = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    outs = {s: tuple(host(t) for t in api.decode(q, kc, vc, num_splits=s, scale=scale,
                                                  with_lse=True))
            for s in (1, 2, 4, 8, 16)}
    Q = host(q)
    for b in range(w.B):
        Kb, Vb = host(kc[b]), host(vc[b])
        for h in range(w.H):
            o_ref, lse_ref = orc.attention_decode(Q[b, h], Kb[h], Vb[h], scale)
            for s, (o, lse) in outs.items():
                assert_close_bf16(o[b, h], lse[b, h], o_ref, lse_ref, f"({b},{h}) splits={s}")


def test_gqa_decode_b64_hq32_hkv8_l32768_every_head():
    w = inputs.GQA_DECODE_L32K
    q, kc, vc = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    outs = {s: tuple(host(t) for t in api.decode(q, kc, vc, num_splits=s, scale=scale,
                                                  with_lse=True))
            for s in (1, 2, 4, 8)}
    Q = host(q)
    for b in range(w.B):
        Kb, Vb = host(kc[b:b + 1]), host(vc[b:b + 1])
        o_ref, lse_ref = orc.attention_decode_gqa(Q[b:b + 1], Kb, Vb, scale)
        for s, (o, lse) in outs.items():
            for h in range(w.H):
                assert_close_bf16(o[b, h], lse[b, h], o_ref[0, h], lse_ref[0, h],
                                  f"({b},{h}) splits={s}")


def test_window_n8192_every_element():
    w = inputs.WINDOW_N8192
    q, k, v = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    o, lse = api.forward(q, k, v, causal=True, scale=scale, window=w.window)
    Q, K, V, O, LSE = (host(t) for t in (q, k, v, o, lse))
    rows = np.arange(w.N)
    for h in range(w.H):
        o_ref, lse_ref = orc.attention_forward_rows(Q[0, h], K[0, h], V[0, h], rows, scale,
                                                    True, window=w.window)
        assert_close_bf16(O[0, h], LSE[0, h], o_ref, lse_ref, f"head {h}")


def test_gqa_train_b8_hq32_hkv8_n4096_every_group():
    w = inputs.GQA_TRAIN_N4096
    q, k, v, do = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    o, lse = api.forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True, scale=scale)
    Q, K, V, DO, O, LSE, DQ, DK, DV = (host(t) for t in (q, k, v, do, o, lse, dq, dk, dv))
    g = w.H // w.kv_heads
    for b, t in ((b, t) for b in range(w.B) for t in range(w.kv_heads)):
        hs = slice(t * g, (t + 1) * g)
        args = (Q[b:b + 1, hs], K[b:b + 1, t:t + 1], V[b:b + 1, t:t + 1])
        o_ref, lse_ref = orc.attention_forward_gqa(*args, scale, True)
        assert_close_bf16(O[b:b + 1, hs], LSE[b:b + 1, hs], o_ref, lse_ref, f"fwd ({b},{t})")
        refs = orc.attention_backward_gqa(*args, DO[b:b + 1, hs], scale, True)
        for name, got, ref in zip(("dq", "dk", "dv"),
                                  (DQ[b:b + 1, hs], DK[b:b + 1, t:t + 1], DV[b:b + 1, t:t + 1]),
                                  refs):
            err = float(np.abs(f64(got) - ref).max())
            assert err <= G_MAX, f"{name} ({b},{t}) max err {err:.3e}"
