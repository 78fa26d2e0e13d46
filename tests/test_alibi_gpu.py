"""ALiBi (bias -slope_h |i - j| on the scaled scores) against the oracle:
forward and backward in bf16, with grouped heads and windows, and the FP8
forward.  Tolerances as for the paths without the bias (bf16: max 2e-2 /
mean 2e-3 on O, 1e-3 on LSE, 5e-2 on gradients)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
import oracle.fp8 as f8
from exact_attention_84_gb300 import api, inputs
from gpu_common import G_MAX, assert_close_bf16, guarded, guards_intact, np64, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu

D = 128
SCALE = 1 / math.sqrt(D)


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 4, 4, 300), (2, 4, 2, 129), (1, 8, 2, 640),
                                        (1, 2, 1, 1)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 150)])
def test_alibi_forward(B, Hq, Hkv, N, causal, window):
    q, k, v = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 100 + N, "cuda")
    slopes = inputs.alibi_slopes(Hq, "cuda")
    bo, o = guarded((B, Hq, N, D), torch.bfloat16)
    bl, lse = guarded((B, Hq, N), torch.float32)
    api.forward(q, k, v, causal=causal, scale=SCALE, out=o, lse=lse, window=window,
                alibi_slopes=slopes)
    o_ref, lse_ref = orc.attention_forward_gqa(np64(q), np64(k), np64(v), SCALE, causal,
                                               window or None, np64(slopes))
    assert_close_bf16(o, lse, o_ref, lse_ref, f"N={N} causal={causal} w={window}")
    assert guards_intact(bo) and guards_intact(bl)


def test_alibi_steep_slope_is_diagonal():
    """A slope of 1e4 leaves only key i for query i: O = V exactly up to the
    bf16 rounding of the output."""
    q, k, v = inputs.gqa_inputs(1, 2, 2, 260, D, torch.bfloat16, 5, "cuda")
    slopes = torch.full((2,), 1e4, device="cuda")
    o, _ = api.forward(q, k, v, causal=False, scale=SCALE, alibi_slopes=slopes)
    assert (o.float() - v.float()).abs().max().item() <= 1e-2


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 2, 2, 200), (2, 4, 2, 256), (1, 4, 1, 130)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 70)])
def test_alibi_backward(B, Hq, Hkv, N, causal, window):
    q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 110 + N, "cuda",
                                    with_do=True)
    slopes = inputs.alibi_slopes(Hq, "cuda")
    o, lse = api.forward(q, k, v, causal=causal, scale=SCALE, window=window, alibi_slopes=slopes)
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=causal, scale=SCALE, window=window,
                              alibi_slopes=slopes)
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), SCALE, causal,
                                      window or None, np64(slopes))
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(np64(got) - ref).max()
        assert err <= G_MAX, f"{name} max err {err:.3e} (N={N} causal={causal} w={window})"


def test_alibi_fp8_forward():
    """FP8 inputs with ALiBi: the element-wise FP8 bound of test_fp8_gpu."""
    B, H, N = 1, 4, 384
    q8, k8, v8 = inputs.fp8_inputs(B, H, H, N, D, 13, "cuda")
    slopes = inputs.alibi_slopes(H, "cuda")
    ds = 1 / inputs.FP8_AMP
    o, lse = api.forward_fp8(q8, k8, v8, ds, ds, ds, causal=True, scale=SCALE,
                             alibi_slopes=slopes)
    q8n, k8n, v8n = (t.cpu().numpy() for t in (q8, k8, v8))
    sl = np64(slopes)
    o_ref, lse_ref = f8.attention_forward_fp8(q8n, k8n, v8n, SCALE, ds, ds, ds, True, None, sl)
    err = np.abs(np64(o) - o_ref)
    for h in range(H):
        # the same bound, with the exact weights taken from the biased scores
        qd = f8.decode_e4m3(q8n[0, h]) * ds
        kd = f8.decode_e4m3(k8n[0, h]) * ds
        vd = f8.decode_e4m3(v8n[0, h])
        bound, _ = fp8_bound_biased(qd, kd, vd, o_ref[0, h], SCALE, sl[h], ds)
        assert (err[0, h] <= bound).all(), f"head {h}: x{(err[0, h] / bound).max():.2f}"
    assert np.abs(np64(lse) - lse_ref).max() <= 1e-3


def fp8_bound_biased(qd, kd, vd, o_ref, scale, slope, v_descale):
    """The FP8 bound of test_fp8_gpu (causal) with the ALiBi bias in the
    scores."""
    n = qd.shape[0]
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    s = (qd @ kd.T) * scale - slope * np.abs(i - j)
    vis = j <= i
    s = np.where(vis, s, -np.inf)
    w = np.where(vis, np.exp(s - s.max(axis=1, keepdims=True)), 0.0)
    l = w.sum(axis=1, keepdims=True)
    p = w / l
    av = np.abs(vd)
    bound = (v_descale * (2.0 ** -4 * (p @ av) + 2.0 ** -10 * (vis @ av) / l)
             + 2.0 ** -8 * np.abs(o_ref) + 1e-4)
    return bound, None


def test_alibi_long_causal_n8192_sampled():
    w = inputs.LONG_CAUSAL
    q, k, v = inputs.workload_inputs(w, "cuda")
    slopes = inputs.alibi_slopes(w.H, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE, alibi_slopes=slopes)
    rng = np.random.default_rng(12)
    rows = np.unique(np.concatenate([np.arange(32), np.arange(w.N - 32, w.N),
                                     rng.choice(w.N, 128, replace=False)]))
    sl = np64(slopes)
    for h in (0, 15, 31):
        o_ref, lse_ref = orc.attention_forward_rows(np64(q[0, h, rows]), np64(k[0, h]),
                                                    np64(v[0, h]), rows, SCALE, True,
                                                    slope=float(sl[h]))
        assert_close_bf16(o[0, h, rows], lse[0, h, rows], o_ref, lse_ref, f"head {h}")


@pytest.mark.parametrize("B,Hq,Hkv,L,splits", [
    (B, Hq, Hkv, L, s)
    for (B, Hq, Hkv, L) in [(2, 4, 4, 1000), (1, 8, 2, 513), (2, 32, 1, 300), (1, 2, 2, 1)]
    for s in [1, 3] if s <= L])
def test_alibi_decode(B, Hq, Hkv, L, splits):
    """Decode with ALiBi: the new token at position L - 1 (both decode
    kernels: one query head per cache head, and grouped heads)."""
    q, kc, vc = inputs.decode_gqa_inputs(B, Hq, Hkv, L, D, torch.bfloat16, 130 + L, "cuda")
    slopes = inputs.alibi_slopes(Hq, "cuda")
    o, lse = api.decode(q, kc, vc, num_splits=splits, scale=SCALE, with_lse=True,
                        alibi_slopes=slopes)
    o_ref, lse_ref = orc.attention_decode_gqa(np64(q), np64(kc), np64(vc), SCALE, np64(slopes))
    assert_close_bf16(o, lse, o_ref, lse_ref, f"L={L} g={Hq // Hkv} splits={splits}")
