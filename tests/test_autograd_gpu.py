"""The autograd wrapper gives the library's forward and gradients inside a
torch.autograd graph (compared with the oracle)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import api, inputs
from gpu_common import G_MAX, O_MAX, np64, status_clean  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,causal,window", [(2, 2, True, 0), (4, 2, True, 50),
                                                  (2, 1, False, 0)])
def test_autograd_matches_oracle(Hq, Hkv, causal, window):
    N, d = 200, 128
    q, k, v, do = inputs.gqa_inputs(1, Hq, Hkv, N, d, torch.bfloat16, 31, "cuda", with_do=True)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = api.attention(qq, kk, vv, causal=causal, window=window)
    (o.float() * do.float()).sum().backward()
    scale = 1 / math.sqrt(d)
    o_ref, _ = orc.attention_forward_gqa(np64(q), np64(k), np64(v), scale, causal, window or None)
    assert np.abs(np64(o) - o_ref).max() <= O_MAX
    refs = orc.attention_backward_gqa(np64(q), np64(k), np64(v), np64(do), scale, causal,
                                      window or None)
    for got, ref in zip((qq.grad, kk.grad, vv.grad), refs):
        assert np.abs(np64(got) - ref).max() <= G_MAX
