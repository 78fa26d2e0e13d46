"""The FP8 (E4M3) part of the oracle against the format's definition, closed
forms and PyTorch's float8_e4m3fn decoding (CPU only), plus planted mistakes
that those pins must catch."""

import math
import os
import types

import numpy as np
import pytest

import oracle.attention as orc
import oracle.fp8 as f8

SRC = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "fp8.py")).read()


def pin_e4m3_closed_forms(m):
    """Values fixed by the E4M3 bit layout (bias 7, 3 mantissa bits)."""
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2 ** -6,
            0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x77: 240.0, 0x78: 256.0, 0x7E: 448.0,
            0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    got = m.decode_e4m3(np.array(list(want), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(want.values()))), got
    nan = m.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()
    # 126 positive finite codes, strictly increasing; within a binade the
    # step is 2^(e-10), and 8 subnormal steps of 2^-9 reach the first normal
    pos = m.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    for code in range(8, 0x7E):
        e = code >> 3
        assert pos[code + 1] - pos[code] == (2.0 ** (e - 10) if (code + 1) >> 3 == e
                                             else 2.0 ** (e - 10))
    # sign bit mirrors every code
    assert np.array_equal(m.decode_e4m3(np.arange(0x80, 0xFF, dtype=np.uint8)),
                          -m.decode_e4m3(np.arange(0x00, 0x7F, dtype=np.uint8)))


def pin_e4m3_torch(m):
    """Library special case: PyTorch's float8_e4m3fn decodes all 256 codes alike."""
    import torch

    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = m.decode_e4m3(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


def pin_fp8_forward(m):
    """The FP8 forward is the pinned definition on the decoded inputs: the
    descale factors act only through their products with the data."""
    r = np.random.default_rng(81)
    B, Hq, Hkv, N, d = 1, 4, 2, 19, 8
    q8, k8, v8 = (r.integers(0, 256, size=s, dtype=np.uint8)
                  for s in ((B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d)))
    for t in (q8, k8, v8):          # keep finite codes only
        t[(t & 0x7F) == 0x7F] = 0x38
        t[(t >> 3 & 0xF) >= 9] &= 0xC7   # keep magnitudes modest (exponent <= 8)
    base_o, base_l = m.attention_forward_fp8(q8, k8, v8, 0.3, 1.0, 1.0, 1.0, True)
    dq, dk, dv = (m.decode_e4m3(t) for t in (q8, k8, v8))
    o_ref, l_ref = orc.attention_forward_gqa(dq, dk, dv, 0.3, True)
    assert np.abs(base_o - o_ref).max() < 1e-14 and np.abs(base_l - l_ref).max() < 1e-14
    # scale * q_descale * k_descale is all that enters the scores
    o2, l2 = m.attention_forward_fp8(q8, k8, v8, 0.3, 2.0, 0.5, 1.0, True)
    assert np.abs(o2 - base_o).max() < 1e-13 and np.abs(l2 - base_l).max() < 1e-13
    o3, l3 = m.attention_forward_fp8(q8, k8, v8, 0.15, 2.0, 1.0, 1.0, True)
    assert np.abs(o3 - base_o).max() < 1e-13 and np.abs(l3 - base_l).max() < 1e-13
    o4, l4 = m.attention_forward_fp8(q8, k8, v8, 0.3, 1.0, 3.0, 1.0, False)
    o5, l5 = m.attention_forward_fp8(q8, k8, v8, 0.9, 1.0, 1.0, 1.0, False)
    assert np.abs(o4 - o5).max() < 1e-13 and np.abs(l4 - l5).max() < 1e-13
    # v_descale scales O and leaves LSE alone
    o6, l6 = m.attention_forward_fp8(q8, k8, v8, 0.3, 1.0, 1.0, 2.5, True)
    assert np.abs(o6 - 2.5 * base_o).max() < 1e-13 and np.abs(l6 - base_l).max() < 1e-15
    # V all 1.0 (code 0x38) -> O = v_descale everywhere
    ones = np.full_like(v8, 0x38)
    o7, _ = m.attention_forward_fp8(q8, k8, ones, 0.3, 1.0, 1.0, 0.75, True)
    assert np.abs(o7 - 0.75).max() < 1e-15
    # causal row 0 sees key 0 only: O_0 = v_descale * V_0, LSE_0 = s_00
    o8, l8 = m.attention_forward_fp8(q8, k8, v8, 0.3, 1.0, 2.0, 1.5, True)
    g = Hq // Hkv
    for h in range(Hq):
        assert np.abs(o8[0, h, 0] - 1.5 * dv[0, h // g, 0]).max() < 1e-15
        assert abs(l8[0, h, 0] - 0.3 * 2.0 * float(dq[0, h, 0] @ dk[0, h // g, 0])) < 1e-13


FP8_PINS = [pin_e4m3_closed_forms, pin_e4m3_torch, pin_fp8_forward]


@pytest.mark.parametrize("pin", FP8_PINS, ids=lambda p: p.__name__)
def test_fp8_pin(pin):
    pin(f8)


MUTANTS = {
    "bias_8": ("np.exp2(exp - 7.0)", "np.exp2(exp - 8.0)"),
    "no_implicit_one": ("(1.0 + man / 8.0)", "(0.5 + man / 8.0)"),
    "subnormal_scale": ("(man / 8.0) * 2.0 ** -6", "(man / 8.0) * 2.0 ** -7"),
    "mantissa_4_bits": ("man = c & 0x7", "man = c & 0xF"),
    "nan_everywhere_in_top_binade": ("(exp == 0xF) & (man == 0x7)", "(exp == 0xF)"),
    "sign_ignored": ("sign = np.where(c & 0x80, -1.0, 1.0)", "sign = np.ones(c.shape)"),
    "v_descale_on_k": ("k = decode_e4m3(k8) * k_descale", "k = decode_e4m3(k8) * v_descale"),
    "q_descale_dropped": ("q = decode_e4m3(q8) * q_descale", "q = decode_e4m3(q8)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_fp8_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = SRC.replace(old, new).replace("from .attention import", "from oracle.attention import")
    mod = types.ModuleType("fp8_mutant")
    exec(compile(src, "fp8_mutant", "exec"), mod.__dict__)
    caught = []
    for pin in FP8_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"
