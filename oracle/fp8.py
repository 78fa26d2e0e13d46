"""FP8 (E4M3) inputs for the fp64 oracle.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may call it.

The pages name FP8 only as a hardware lever of FlashAttention-3
("03. FlashAttention", section "FlashAttention v3"); they do not define a
format.  The reading taken is the OCP 8-bit floating-point E4M3 format:
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
holds the subnormals m/8 * 2^-6; the all-ones exponent is an ordinary
binade except mantissa 7, which is NaN (no infinities).  A tensor's real
values are its codes decoded times a per-tensor descale factor.

* ``decode_e4m3`` -- codes (uint8) -> float64, from the bit fields above.
* ``attention_forward_fp8`` -- the attention definition of
  ``attention.attention_forward_gqa`` evaluated on the decoded, descaled
  inputs.  FP8 changes only what the inputs are; the method stays exact
  ("03. FlashAttention", "Benefices"), so the oracle is the same
  definition.  The GPU additionally rounds P to E4M3 before P.V; that
  rounding is an error of the kernel, bounded in the tests, not part of
  the definition.

Pins: tests/oracle_pins.py (pin_e4m3_decode, pin_fp8_forward).
"""

from __future__ import annotations

import numpy as np

from .attention import attention_forward_gqa

__all__ = ["decode_e4m3", "attention_forward_fp8"]


def decode_e4m3(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = (1.0 + man / 8.0) * np.exp2(exp - 7.0)
    subnormal = (man / 8.0) * 2.0 ** -6
    val = sign * np.where(exp == 0, subnormal, normal)
    return np.where((exp == 0xF) & (man == 0x7), np.nan, val)


def attention_forward_fp8(q8, k8, v8, scale: float, q_descale: float, k_descale: float,
                          v_descale: float, causal: bool, window=None, alibi_slopes=None):
    """q8 [B, Hq, N, d], k8/v8 [B, Hkv, N, d] E4M3 codes -> (O, LSE) of
    attention over Q = q_descale*decode(q8), K = k_descale*decode(k8),
    V = v_descale*decode(v8)."""
    q = decode_e4m3(q8) * q_descale
    k = decode_e4m3(k8) * k_descale
    v = decode_e4m3(v8) * v_descale
    return attention_forward_gqa(q, k, v, scale, causal, window, alibi_slopes)
