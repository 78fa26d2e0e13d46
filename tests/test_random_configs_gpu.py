"""Seeded random configurations of the whole path against the oracle: batch,
query and key/value head counts, sequence lengths that hit every tile
remainder, the causal mask, windows, ALiBi and the deterministic backward
drawn together, with guarded outputs.  Decode draws cache lengths and split
counts the same way.  Tolerances as elsewhere (O max 2e-2 / mean 2e-3, LSE
1e-3, gradients 5e-2 against the oracle's exact-O gradients) for every draw
at the workloads' scale 1/sqrt(d) or below (0.05).  The draws at scale 0.2
(2.3 times 1/sqrt(d)) have peaked rows with gradients of magnitude ~10-30: a
bf16 result is then off by up to half a unit in its last place, 2^-8 |g|,
before any arithmetic, so there each gradient element may also differ by
2^-7 |g_ref| (that rounding plus as much again for the bf16 P and dS
operands), and D = rowsum(dO * O) is formed from the O the forward stored,
as the kernel forms it (where dP - D cancels in a nearly one-hot row, the
rounding of O to bf16 moves D by more than the gradient tolerance)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import api, inputs
from gpu_common import G_MAX, assert_close_bf16, guarded, guards_intact, np64, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu

D = 128


def draw(seed):
    r = np.random.default_rng(1000 + seed)
    hkv = int(r.choice([1, 2, 3]))
    g = int(r.choice([1, 2, 4]))
    N = int(r.integers(1, 700))
    causal = bool(r.integers(0, 2))
    window = int(r.integers(1, N + 80)) if causal and r.random() < 0.5 else 0
    alibi = bool(r.random() < 0.35)
    scale = float(r.choice([1 / math.sqrt(D), 0.05, 0.2]))
    det = bool(r.random() < 0.3)
    return dict(B=int(r.integers(1, 3)), Hq=hkv * g, Hkv=hkv, N=N, causal=causal, window=window,
                alibi=alibi, scale=scale, det=det)


@pytest.mark.parametrize("seed", range(48))
def test_random_forward_backward(seed):
    c = draw(seed)
    B, Hq, Hkv, N = c["B"], c["Hq"], c["Hkv"], c["N"]
    q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 500 + seed, "cuda",
                                    with_do=True)
    slopes = inputs.alibi_slopes(Hq, "cuda") if c["alibi"] else None
    bo, o = guarded((B, Hq, N, D), torch.bfloat16)
    bl, lse = guarded((B, Hq, N), torch.float32)
    api.forward(q, k, v, causal=c["causal"], scale=c["scale"], out=o, lse=lse,
                window=c["window"], alibi_slopes=slopes)
    sl = None if slopes is None else np64(slopes)
    win = c["window"] or None
    o_ref, lse_ref = orc.attention_forward_gqa(np64(q), np64(k), np64(v), c["scale"], c["causal"],
                                               win, sl)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"{c}")
    assert guards_intact(bo) and guards_intact(bl)
    bq, dq = guarded((B, Hq, N, D), torch.bfloat16)
    bk, dk = guarded((B, Hkv, N, D), torch.bfloat16)
    bv, dv = guarded((B, Hkv, N, D), torch.bfloat16)
    api.backward(q, k, v, o, lse, do, causal=c["causal"], scale=c["scale"], out=(dq, dk, dv),
                 window=c["window"], alibi_slopes=slopes, deterministic=c["det"])
    plain = c["scale"] <= 1 / math.sqrt(D) + 1e-12
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), c["scale"],
                                      c["causal"], win, sl, o=None if plain else np64(o))
    rel = 0.0 if plain else 2.0 ** -7
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(np64(got) - ref)
        over = (err / (G_MAX + rel * np.abs(ref))).max()
        assert over <= 1.0, f"{name} max err {err.max():.3e} (x{over:.2f} of the bound) {c}"
    assert guards_intact(bq) and guards_intact(bk) and guards_intact(bv)


@pytest.mark.parametrize("seed", range(24))
def test_random_decode(seed):
    r = np.random.default_rng(2000 + seed)
    hkv = int(r.choice([1, 2, 4]))
    g = int(r.choice([1, 2, 4, 8]))
    B, Hq, L = int(r.integers(1, 4)), hkv * g, int(r.integers(1, 5000))
    splits = int(r.choice([0, 1, 2, 3, 8]))
    splits = min(splits, L) if splits else 0
    alibi = bool(r.random() < 0.3)
    q, kc, vc = inputs.decode_gqa_inputs(B, Hq, hkv, L, D, torch.bfloat16, 600 + seed, "cuda")
    slopes = inputs.alibi_slopes(Hq, "cuda") if alibi else None
    o, lse = api.decode(q, kc, vc, num_splits=splits, scale=1 / math.sqrt(D), with_lse=True,
                        alibi_slopes=slopes)
    o_ref, lse_ref = orc.attention_decode_gqa(np64(q), np64(kc), np64(vc), 1 / math.sqrt(D),
                                              None if slopes is None else np64(slopes))
    assert_close_bf16(o, lse, o_ref, lse_ref, f"B={B} Hq={Hq} Hkv={hkv} L={L} splits={splits}")
