"""bf16 tcgen05 forward against the oracle (max 2e-2, mean 2e-3 on O; 1e-3 on LSE)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import (G_MAX, FP32_TOL, LSE_MAX, O_MAX, assert_close_bf16, guarded,
                        guards_intact, np64, status_clean)  # noqa: F401

pytestmark = pytest.mark.gpu

# ------------------------------------------------------------- bf16 forward
@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 1, 128), (1, 2, 129), (2, 3, 300),
                                   (1, 1, 640), (1, 2, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_forward_shapes(B, H, N, causal):
    d = 128
    q, k, v = inputs.attention_inputs(B, H, N, d, torch.bfloat16, 20 + N, "cuda")
    scale = 1 / math.sqrt(d)
    bo, o = guarded((B, H, N, d), torch.bfloat16)
    bl, lse = guarded((B, H, N), torch.float32)
    api.forward(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), scale, causal)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"N={N} causal={causal}")
    assert guards_intact(bo) and guards_intact(bl)


def test_bf16_forward_other_scale():
    q, k, v = inputs.attention_inputs(1, 2, 256, 128, torch.bfloat16, 77, "cuda")
    o, lse = api.forward(q, k, v, causal=True, scale=0.02)
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), 0.02, True)
    assert_close_bf16(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_forward_b4_h16_n2048(causal):
    w = inputs.FWD_N2048
    q, k, v = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale)
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), scale, causal)
    assert_close_bf16(o, lse, o_ref, lse_ref, f"causal={causal}")


def test_bf16_forward_split_tail_items_ragged_gqa():
    """Non-causal, 160 (Q pair, head) items on 152 SMs: the last 8 items run
    as 16 one-tile blocks.  They are the last Q pair (tiles 18 and 19, the
    second past N = 2500) of query heads 8..15; check those rows and others
    against the oracle, and that nothing is written past O's end."""
    B, Hq, Hkv, N, D = 1, 16, 4, 2500, 128
    q, k, v = inputs.gqa_inputs(B, Hq, Hkv, N, D, torch.bfloat16, 77, "cuda")
    scale = 1 / math.sqrt(D)
    bo, o = guarded((B, Hq, N, D), torch.bfloat16)
    bl, lse = guarded((B, Hq, N), torch.float32)
    api.forward(q, k, v, causal=False, scale=scale, out=o, lse=lse)
    rng = np.random.default_rng(77)
    rows = np.unique(np.concatenate([np.arange(2304, N), rng.choice(2304, 64, replace=False)]))
    for h in (0, 8, 11, 15):
        t = h // (Hq // Hkv)
        o_ref, lse_ref = orc.attention_forward_rows(np64(q[0, h, rows]), np64(k[0, t]),
                                                    np64(v[0, t]), rows, scale, False)
        assert_close_bf16(o[0, h, rows], lse[0, h, rows], o_ref, lse_ref, f"head {h}")
    assert guards_intact(bo) and guards_intact(bl)
