"""bf16 backward (dQ, dK, dV) against the oracle's analytic gradient (max 5e-2)."""
import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs
from gpu_common import (G_MAX, FP32_TOL, LSE_MAX, O_MAX, assert_close_bf16, guarded,
                        guards_intact, np64, status_clean)  # noqa: F401

pytestmark = pytest.mark.gpu

# ------------------------------------------------------------ bf16 backward
@pytest.mark.parametrize("B,H,N", [(1, 1, 64), (1, 2, 200), (2, 2, 256), (1, 1, 1),
                                   (1, 1, 130), (1, 2, 520)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_shapes(B, H, N, causal):
    d = 128
    q, k, v, do = inputs.attention_inputs(B, H, N, d, torch.bfloat16, 30 + N, "cuda",
                                          with_do=True)
    scale = 1 / math.sqrt(d)
    o, lse = api.forward(q, k, v, causal=causal, scale=scale)
    bq, dq = guarded((B, H, N, d), torch.bfloat16)
    bk, dk = guarded((B, H, N, d), torch.bfloat16)
    bv, dv = guarded((B, H, N, d), torch.bfloat16)
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_BACKWARD, B, H, N, d, 0),
                     dtype=torch.uint8, device="cuda")
    _lib.check(_lib.fa_backward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, N, d, scale, int(causal), ws.data_ptr(),
                                   ws.numel(), torch.cuda.current_stream().cuda_stream))
    refs = orc.attention_backward(np64(q), np64(k), np64(v), np64(do), scale, causal)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(np64(got) - ref).max()
        assert err <= G_MAX, f"{name} max err {err:.3e} (N={N}, causal={causal})"
    assert guards_intact(bq) and guards_intact(bk) and guards_intact(bv)


