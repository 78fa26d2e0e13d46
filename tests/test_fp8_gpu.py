"""FP8 (E4M3) forward against the oracle on the decoded inputs.

Tolerance (derived from the kernel's arithmetic, no page states one): the
inputs are the same E4M3 values on both sides, products accumulate in fp32,
and the kernel rounds each unnormalised weight p_j (p_j <= 2^8 in its own
reference frame) to E4M3 before P.V: a relative error of at most 2^-4 for
normal values and an absolute error of at most 2^-10 below 2^-6.  The
normaliser l sums the unrounded weights.  So, per output element,

  |dO_ic| <= v_descale * (2^-4 sum_j P_ij |V_jc| + 2^-10 sum_j |V_jc| / l_i)
             + 2^-8 |O_ic| + 1e-4

with P, V the exact (oracle) weights and decoded values, sum_j over the keys
row i sees, and l_i = sum_j exp(s_ij - max_j s_ij) >= 1 (the kernel's l is
taken relative to a reference no larger than the row maximum, so it is at
least this large).  The last terms cover the bf16 output rounding and fp32
accumulation.

Mean error: rounding to 3 mantissa bits leaves each weight an error spread
over at most one unit in the last place, 2^-3 p_j (2^-9 / l_i in normalised
units below 2^-6), so its standard deviation is at most that over sqrt(12)
and, summed over the keys,

  sigma_ic = v_descale * sqrt(2^-6/12 sum_j P_ij^2 V_jc^2
                              + 2^-18/12 sum_j V_jc^2 / l_i^2).

The mean of |dO| over all elements (about 0.8 sigma for independent
roundings) must not exceed the mean of sigma plus the bf16 output rounding
(2^-9 |O| on average at most).  The bf16 path's 2e-3 does not carry over:
its P keeps 8 mantissa bits.  LSE stays within 1e-3 (l uses unrounded
weights).
"""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
import oracle.fp8 as f8
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import LSE_MAX, guarded, guards_intact, np64, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu

D = 128
SCALE = 1 / math.sqrt(D)
DS = 1 / inputs.FP8_AMP


def fp8_bound(qd, kd, vd, o_ref, scale, causal, window, v_descale, rows=None):
    """Per-element error bound and sigma above, for one head: qd [R, d] the
    query rows at positions `rows` (default: all), kd [N, d] decoded and
    descaled, vd [N, d] decoded (v_descale applied here), o_ref [R, d]."""
    rows = np.arange(qd.shape[0]) if rows is None else np.asarray(rows)
    s = (qd @ kd.T) * scale
    i = rows[:, None]
    j = np.arange(kd.shape[0])[None, :]
    vis = np.ones_like(s, dtype=bool)
    if causal:
        vis &= j <= i
    if window:
        vis &= j > i - window
    s = np.where(vis, s, -np.inf)
    mx = s.max(axis=1, keepdims=True)
    w = np.where(vis, np.exp(s - mx), 0.0)
    l = w.sum(axis=1, keepdims=True)
    p = w / l
    av = np.abs(vd)
    bound = (v_descale * (2.0 ** -4 * (p @ av) + 2.0 ** -10 * (vis @ av) / l)
             + 2.0 ** -8 * np.abs(o_ref) + 1e-4)
    v2 = vd * vd
    sigma = v_descale * np.sqrt(2.0 ** -6 / 12 * ((p * p) @ v2)
                                + 2.0 ** -18 / 12 * (vis @ v2) / (l * l))
    return bound, sigma


def check_fp8(o, lse, q8, k8, v8, scale, causal, window, descales, what):
    qs, ks, vs = descales
    q8n, k8n, v8n = (t.cpu().numpy() for t in (q8, k8, v8))
    o_ref, lse_ref = f8.attention_forward_fp8(q8n, k8n, v8n, scale, qs, ks, vs, causal,
                                              window or None)
    got = np64(o)
    err = np.abs(got - o_ref)
    g = q8.shape[1] // k8.shape[1]
    worst = 0.0
    sig = np.zeros_like(err)
    for b in range(q8.shape[0]):
        for h in range(q8.shape[1]):
            qd = f8.decode_e4m3(q8n[b, h]) * qs
            kd = f8.decode_e4m3(k8n[b, h // g]) * ks
            vd = f8.decode_e4m3(v8n[b, h // g])
            bound, sig[b, h] = fp8_bound(qd, kd, vd, o_ref[b, h], scale, causal, window, vs)
            ratio = (err[b, h] / bound).max()
            worst = max(worst, ratio)
            assert ratio <= 1.0, f"{what} ({b},{h}): error exceeds the bound by x{ratio:.2f}"
    mean_lim = sig.mean() + 2.0 ** -9 * np.abs(o_ref).mean() + 1e-5
    assert err.mean() <= mean_lim, f"{what} mean|dO| = {err.mean():.3e} > {mean_lim:.3e}"
    dl = np.abs(np64(lse) - lse_ref).max()
    assert dl <= LSE_MAX, f"{what} max|dLSE| = {dl:.3e}"
    print(f"{what}: max|dO| {err.max():.3e} mean {err.mean():.3e} (limit {mean_lim:.3e}) "
          f"worst/bound {worst:.3f}")


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 1, 1, 1), (1, 2, 2, 128), (2, 2, 1, 300),
                                        (1, 4, 2, 640), (1, 1, 1, 1000)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 100)])
def test_fp8_forward(B, Hq, Hkv, N, causal, window):
    q8, k8, v8 = inputs.fp8_inputs(B, Hq, Hkv, N, D, 90 + N, "cuda")
    bo, o = guarded((B, Hq, N, D), torch.bfloat16)
    bl, lse = guarded((B, Hq, N), torch.float32)
    api.forward_fp8(q8, k8, v8, DS, DS, DS, causal=causal, scale=SCALE, window=window, out=o,
                    lse=lse)
    check_fp8(o, lse, q8, k8, v8, SCALE, causal, window, (DS, DS, DS),
              f"N={N} causal={causal} w={window}")
    assert guards_intact(bo) and guards_intact(bl)


def test_fp8_forward_descales_and_workspace():
    """Unequal descale factors, and a caller-owned workspace."""
    B, H, N = 1, 2, 520
    q8, k8, v8 = inputs.fp8_inputs(B, H, H, N, D, 7, "cuda", amp=4.0)
    nbytes = _lib.fa_workspace_size(_lib.FA_OP_FORWARD_FP8, B, H, N, D, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    qs, ks, vs = 0.25, 0.5, 2.0
    o, lse = api.forward_fp8(q8, k8, v8, qs, ks, vs, causal=True, scale=0.1, workspace=ws)
    check_fp8(o, lse, q8, k8, v8, 0.1, True, 0, (qs, ks, vs), "descales")


def test_fp8_uniform_v():
    """All V codes 1.0: O = v_descale within the bound, and exactly so in
    row 0 of a causal pass (one key, weight 1)."""
    B, H, N = 1, 2, 384
    q8, k8, _ = inputs.fp8_inputs(B, H, H, N, D, 11, "cuda")
    v8 = torch.full_like(q8, 0x38)
    o, lse = api.forward_fp8(q8, k8, v8, DS, DS, 0.5, causal=True, scale=SCALE)
    assert (o[:, :, 0].float() - 0.5).abs().max().item() == 0.0
    check_fp8(o, lse, q8, k8, v8, SCALE, True, 0, (DS, DS, 0.5), "uniform V")


def test_fp8_long_causal_n8192_every_element():
    """The fp8 workload (B1 H32 N8192, causal) in full: every element of
    every head within the bound above, the mean over all of them within the
    mean limit, every LSE within 1e-3.  Head by head, so the host holds one
    8192 x 8192 score matrix at a time."""
    w = inputs.FP8_LONG_CAUSAL
    q8, k8, v8 = inputs.workload_inputs(w, "cuda")
    o, lse = api.forward_fp8(q8, k8, v8, DS, DS, DS, causal=True, scale=SCALE)
    O, LSE = np64(o), np64(lse)
    q8n, k8n, v8n = (t.cpu().numpy() for t in (q8, k8, v8))
    err_sum = sig_sum = ref_sum = 0.0
    for h in range(w.H):
        sl = slice(h, h + 1)
        o_ref, lse_ref = f8.attention_forward_fp8(q8n[:, sl], k8n[:, sl], v8n[:, sl], SCALE,
                                                  DS, DS, DS, True, None)
        qd = f8.decode_e4m3(q8n[0, h]) * DS
        kd = f8.decode_e4m3(k8n[0, h]) * DS
        vd = f8.decode_e4m3(v8n[0, h])
        err = np.abs(O[0, h] - o_ref[0, 0])
        bound, sig = fp8_bound(qd, kd, vd, o_ref[0, 0], SCALE, True, 0, DS)
        assert (err <= bound).all(), f"head {h}: x{(err / bound).max():.2f} over the bound"
        assert np.abs(LSE[0, h] - lse_ref[0, 0]).max() <= LSE_MAX, f"head {h} LSE"
        err_sum += err.sum()
        sig_sum += sig.sum()
        ref_sum += np.abs(o_ref).sum()
    n = O.size
    assert err_sum / n <= sig_sum / n + 2.0 ** -9 * ref_sum / n + 1e-5
