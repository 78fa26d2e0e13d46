"""Shared helpers of the GPU parity tests: the CUDA path (through the C-ABI)
against the fp64 oracle on the same bytes.

Tolerances: fp32 path max|dO| <= 1e-5 on O and LSE; bf16 path (fp32
accumulation) max|dO| <= 2e-2, mean|dO| <= 2e-3, max|dLSE| <= 1e-3 and
max|d grad| <= 5e-2.  Small shapes are compared element by element (several
tiles plus a ragged tail); the full-size workloads run in the launch
configuration the bench times and are compared element by element too
(tests/test_full_workloads_gpu.py).
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as orc
from exact_attention_84_gb300 import _lib, api, inputs

O_MAX, O_MEAN, LSE_MAX, G_MAX = 2e-2, 2e-3, 1e-3, 5e-2
FP32_TOL = 1e-5


def np64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def assert_close_bf16(o, lse, o_ref, lse_ref, what=""):
    d = np.abs(np64(o) - o_ref)
    assert d.max() <= O_MAX, f"{what} max|dO| = {d.max():.3e}"
    assert d.mean() <= O_MEAN, f"{what} mean|dO| = {d.mean():.3e}"
    if lse is not None:
        dl = np.abs(np64(lse) - lse_ref)
        assert dl.max() <= LSE_MAX, f"{what} max|dLSE| = {dl.max():.3e}"


def guarded(shape, dtype, pad=256):
    """A contiguous tensor of `shape` inside a larger buffer whose guard bands
    are filled with a sentinel, so out-of-bounds writes can be detected."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), 12345.0, dtype=dtype, device="cuda")
    view = buf[pad:pad + n].view(shape)
    return buf, view


def guards_intact(buf, pad=256):
    lo, hi = buf[:pad], buf[-pad:]
    return bool((lo == 12345.0).all() and (hi == 12345.0).all())


@pytest.fixture(autouse=True)
def status_clean():
    yield
    assert api.device_status() == 0, _lib.fa_last_error()


