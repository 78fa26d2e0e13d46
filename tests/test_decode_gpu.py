"""Split-KV decode against the unsplit oracle, for several split counts."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import (G_MAX, FP32_TOL, LSE_MAX, O_MAX, assert_close_bf16, guarded,
                        guards_intact, np64, status_clean)  # noqa: F401

pytestmark = pytest.mark.gpu

# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("B,H,L", [(1, 1, 1), (2, 3, 1000), (1, 2, 4097), (3, 1, 64)])
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16])
def test_decode_shapes(B, H, L, splits):
    if splits > L:
        pytest.skip("num_splits > Lkv is rejected by the API")
    d = 128
    q, kc, vc = inputs.decode_inputs(B, H, L, d, torch.bfloat16, 40 + L, "cuda")
    scale = 1 / math.sqrt(d)
    o, lse = api.decode(q, kc, vc, num_splits=splits, scale=scale, with_lse=True)
    o_ref, lse_ref = orc.attention_decode(np64(q), np64(kc), np64(vc), scale)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"L={L} splits={splits}")


def test_decode_default_entry_point():
    q, kc, vc = inputs.decode_inputs(2, 2, 777, 128, torch.bfloat16, 5, "cuda")
    o = api.decode(q, kc, vc, num_splits=5)
    o_ref, _ = orc.attention_decode(np64(q), np64(kc), np64(vc), 1 / math.sqrt(128))
    assert_close_bf16(o, None, o_ref, None)


def test_decode_b64_h32_l32768_sampled():
    w = inputs.DECODE_L32K
    q, kc, vc = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    outs = {s: api.decode(q, kc, vc, num_splits=s, scale=scale, with_lse=True)
            for s in (1, 4, 16)}
    rng = np.random.default_rng(4)
    pairs = [(0, 0), (w.B - 1, w.H - 1)] + [tuple(x) for x in
                                            zip(rng.integers(0, w.B, 6), rng.integers(0, w.H, 6))]
    for b, h in pairs:
        o_ref, lse_ref = orc.attention_decode(np64(q[b, h]), np64(kc[b, h]), np64(vc[b, h]),
                                              scale)
        for s, (o, lse) in outs.items():
            assert_close_bf16(o[b, h], lse[b, h], o_ref, lse_ref, f"({b},{h}) splits={s}")
    # split invariance over every (b, h): the parts recombine to the same answer
    o1 = outs[1][0].float()
    for s in (4, 16):
        assert (outs[s][0].float() - o1).abs().max().item() <= 2 * O_MAX
        assert (outs[s][1] - outs[1][1]).abs().max().item() <= LSE_MAX
