"""fp32 forward (true fp32 FMA) against the oracle: max|dO|, max|dLSE| <= 1e-5."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import (G_MAX, FP32_TOL, LSE_MAX, O_MAX, assert_close_bf16, guarded,
                        guards_intact, np64, status_clean)  # noqa: F401

pytestmark = pytest.mark.gpu

# ----------------------------------------------------------------- fp32 path
def test_fp32_tiny_workload():
    w = inputs.TINY_FP32
    q, k, v = inputs.workload_inputs(w, "cuda")
    scale = 1 / math.sqrt(w.d)
    o, lse = api.forward(q, k, v, causal=False, scale=scale)
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), scale, False)
    assert np.abs(np64(o) - o_ref).max() <= FP32_TOL
    assert np.abs(np64(lse) - lse_ref).max() <= FP32_TOL


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 1, 32, False), (2, 1, 7, 64, True),
                                            (1, 1, 129, 128, True), (1, 3, 300, 96, False),
                                            (2, 2, 256, 64, True)])
def test_fp32_shapes(B, H, N, d, causal):
    q, k, v = inputs.attention_inputs(B, H, N, d, torch.float32, 10 + N, "cuda")
    scale = 1 / math.sqrt(d)
    bo, o = guarded((B, H, N, d), torch.float32)
    bl, lse = guarded((B, H, N), torch.float32)
    api.forward(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
    o_ref, lse_ref = orc.attention_forward(np64(q), np64(k), np64(v), scale, causal)
    assert np.abs(np64(o) - o_ref).max() <= FP32_TOL
    assert np.abs(np64(lse) - lse_ref).max() <= FP32_TOL
    assert guards_intact(bo) and guards_intact(bl)


