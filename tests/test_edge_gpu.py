"""Edge cases across the paths: sequence lengths one past or one short of a
tile multiple at larger sizes, the maximum split count, one cache row per
split, and the extensions combined (grouped heads + window + ALiBi +
deterministic backward; FP8 + grouped heads + window)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
import oracle.fp8 as f8
from exact_attention_84_gb300 import api, inputs
from gpu_common import G_MAX, assert_close_bf16, np64, status_clean  # noqa: F401
from test_fp8_gpu import check_fp8

pytestmark = pytest.mark.gpu

D = 128
SCALE = 1 / math.sqrt(D)


@pytest.mark.parametrize("N", [8191, 8193])
def test_forward_ragged_long(N):
    q, k, v = inputs.attention_inputs(1, 2, N, D, torch.bfloat16, N, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(N - 130, N),
                                     np.random.default_rng(N).choice(N, 64, replace=False)]))
    for h in range(2):
        o_ref, lse_ref = orc.attention_forward_rows(np64(q[0, h, rows]), np64(k[0, h]),
                                                    np64(v[0, h]), rows, SCALE, True)
        assert_close_bf16(o[0, h, rows], lse[0, h, rows], o_ref, lse_ref, f"N={N} h={h}")


@pytest.mark.parametrize("deterministic", [False, True])
def test_backward_ragged_1025(deterministic):
    q, k, v, do = inputs.attention_inputs(1, 1, 1025, D, torch.bfloat16, 11, "cuda", with_do=True)
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE)
    grads = api.backward(q, k, v, o, lse, do, causal=True, scale=SCALE,
                         deterministic=deterministic)
    refs = orc.attention_backward(np64(q), np64(k), np64(v), np64(do), SCALE, True)
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        err = np.abs(np64(got) - ref).max()
        assert err <= G_MAX, f"{name} max err {err:.3e}"


@pytest.mark.parametrize("L,splits", [(32769, 1), (32769, 7), (32769, 1024), (64, 64)])
def test_decode_split_extremes(L, splits):
    """Up to the maximum split count, and one cache row per split."""
    q, kc, vc = inputs.decode_inputs(1, 2, L, D, torch.bfloat16, L + splits, "cuda")
    o, lse = api.decode(q, kc, vc, num_splits=splits, scale=SCALE, with_lse=True)
    o_ref, lse_ref = orc.attention_decode(np64(q), np64(kc), np64(vc), SCALE)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"L={L} splits={splits}")


def test_extensions_combined_bf16():
    """Grouped heads, a window and ALiBi together, forward and deterministic
    backward."""
    B, Hq, Hkv, N, W = 2, 6, 2, 333, 77
    q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 21, "cuda", with_do=True)
    sl = inputs.alibi_slopes(Hq, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=SCALE, window=W, alibi_slopes=sl)
    o_ref, lse_ref = orc.attention_forward_gqa(np64(q), np64(k), np64(v), SCALE, True, W,
                                               np64(sl))
    assert_close_bf16(o, lse, o_ref, lse_ref)
    grads = api.backward(q, k, v, o, lse, do, causal=True, scale=SCALE, window=W,
                         alibi_slopes=sl, deterministic=True)
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), SCALE, True, W,
                                      np64(sl))
    for name, got, ref in zip(("dq", "dk", "dv"), grads, refs):
        err = np.abs(np64(got) - ref).max()
        assert err <= G_MAX, f"{name} max err {err:.3e}"


def test_extensions_combined_fp8():
    """FP8 inputs with grouped heads and a window, under the FP8 bound."""
    B, Hq, Hkv, N, W = 1, 4, 2, 300, 90
    q8, k8, v8 = inputs.fp8_inputs(B, Hq, Hkv, N, D, 22, "cuda")
    ds = 1 / inputs.FP8_AMP
    o, lse = api.forward_fp8(q8, k8, v8, ds, ds, ds, causal=True, scale=SCALE, window=W)
    check_fp8(o, lse, q8, k8, v8, SCALE, True, W, (ds, ds, ds), "fp8 gqa window")


@pytest.mark.parametrize("causal", [False, True])
def test_peaked_softmax(causal):
    """Inputs scaled by 8: scores with a standard deviation of about 64, so
    each row's softmax is nearly one-hot and the running maximum jumps by far
    more than the rescale threshold; forward and backward against the
    oracle."""
    B, H, N = 1, 2, 700
    q, k, v, do = inputs.attention_inputs(B, H, N, D, torch.bfloat16, 61, "cuda", with_do=True)
    q, k = (t.float().mul(8.0).to(torch.bfloat16) for t in (q, k))
    o, lse = api.forward(q, k, v, causal=causal, scale=SCALE)
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), SCALE, causal)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"causal={causal}")
    grads = api.backward(q, k, v, o, lse, do, causal=causal, scale=SCALE)
    # The backward forms D = rowsum(dO * O) from the O the forward stored (in
    # bf16); with a nearly one-hot softmax dP - D cancels, so the reference
    # takes the same stored O.  dQ and dK scale linearly with |K| and |Q|
    # (x8 here), so their tolerance is 8 times the unit-scale 5e-2.
    refs = orc.attention_backward(np64(q), np64(k), np64(v), np64(do), SCALE, causal,
                                  o=np64(o))
    for name, got, ref, tol in zip(("dq", "dk", "dv"), grads, refs, (8 * G_MAX, 8 * G_MAX, G_MAX)):
        err = np.abs(np64(got) - ref).max()
        assert err <= tol, f"{name} max err {err:.3e} (tolerance {tol:.2e})"
