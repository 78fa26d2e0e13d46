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
# every split count up to Lkv (more splits than cache rows is rejected by the
# API before any launch, which the host tests check)
@pytest.mark.parametrize("B,H,L,splits", [
    (B, H, L, s) for (B, H, L) in [(1, 1, 1), (2, 3, 1000), (1, 2, 4097), (3, 1, 64)]
    for s in [1, 2, 3, 7, 16] if s <= L])
def test_decode_shapes(B, H, L, splits):
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


