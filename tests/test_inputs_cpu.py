"""The seeded input recipe (CPU): draws are reproducible, have the shapes,
dtypes and structure the workloads name, and the workload table is
self-consistent."""
import math

import pytest
import torch

from exact_attention_84_gb300 import inputs


def test_same_seed_same_tensors_other_seed_differs():
    a = inputs.attention_inputs(2, 3, 17, 8, torch.bfloat16, 5, "cpu", with_do=True)
    b = inputs.attention_inputs(2, 3, 17, 8, torch.bfloat16, 5, "cpu", with_do=True)
    c = inputs.attention_inputs(2, 3, 17, 8, torch.bfloat16, 6, "cpu", with_do=True)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not any(torch.equal(x, y) for x, y in zip(a, c))
    # Q, K, V, dO are distinct draws, not copies of one another
    assert not torch.equal(a[0], a[1]) and not torch.equal(a[1], a[2])


def test_shapes_and_dtypes():
    q, k, v, do = inputs.gqa_inputs(2, 8, 2, 33, 16, torch.bfloat16, 1, "cpu", with_do=True)
    assert q.shape == (2, 8, 33, 16) and do.shape == q.shape
    assert k.shape == (2, 2, 33, 16) and v.shape == k.shape
    assert {t.dtype for t in (q, k, v, do)} == {torch.bfloat16}
    q, kc, vc = inputs.decode_gqa_inputs(3, 8, 4, 40, 16, torch.bfloat16, 2, "cpu")
    assert q.shape == (3, 8, 16) and kc.shape == (3, 4, 40, 16) and vc.shape == kc.shape
    q, kc, vc = inputs.decode_inputs(3, 4, 40, 16, torch.bfloat16, 2, "cpu")
    assert q.shape == (3, 4, 16) and kc.shape == (3, 4, 40, 16)
    q, k, v = inputs.attention_inputs(1, 1, 9, 4, torch.float32, 0, "cpu")
    assert q.dtype == torch.float32 and q.is_contiguous()


def test_bf16_is_the_fp32_draw_rounded_to_nearest():
    """Each tensor is drawn as fp32 standard normals, batch by batch, then
    rounded to the storage dtype."""
    q16, = inputs.attention_inputs(2, 2, 5, 4, torch.bfloat16, 9, "cpu")[:1]
    g = inputs.generator(9, "cpu")
    ref = torch.stack([torch.randn((2, 5, 4), generator=g, dtype=torch.float32)
                       for _ in range(2)])
    assert torch.equal(q16, ref.to(torch.bfloat16))


def test_uniform_head_has_identical_keys():
    q, k, v = inputs.attention_inputs(2, 3, 11, 4, torch.bfloat16, 4, "cpu", uniform_head=1)
    assert torch.equal(k[:, 1], k[:, 1, :1].expand(-1, 11, -1))
    assert not torch.equal(k[:, 0], k[:, 0, :1].expand(-1, 11, -1))


def test_fp8_codes_stay_in_range():
    q8, k8, v8 = inputs.fp8_inputs(1, 4, 2, 64, 16, 8, "cpu")
    assert q8.dtype == torch.uint8 and q8.shape == (1, 4, 64, 16) and k8.shape == (1, 2, 64, 16)
    for t in (q8, k8, v8):
        x = t.view(torch.float8_e4m3fn).float()
        assert torch.isfinite(x).all()
        assert x.abs().max().item() < 448.0
        # amplified N(0,1) draws: spread over the format, far from all zero
        assert x.std().item() > inputs.FP8_AMP / 2


def test_alibi_slopes_schedule():
    for H in (1, 8, 32):
        s = inputs.alibi_slopes(H, "cpu").double()
        assert s.shape == (H,) and (s > 0).all()
        assert math.isclose(s[0].item(), 2.0 ** (-8.0 / H), rel_tol=1e-6)
        assert math.isclose(s[-1].item(), 2.0 ** -8, rel_tol=1e-6)
        if H > 1:
            ratio = (s[1:] / s[:-1])
            assert torch.allclose(ratio, torch.full_like(ratio, 2.0 ** (-8.0 / H)), rtol=1e-6)


def test_workload_table_is_consistent():
    names = [w.name for w in inputs.ALL]
    seeds = [w.seed for w in inputs.ALL]
    assert len(set(names)) == len(names) and len(set(seeds)) == len(seeds)
    for w in inputs.ALL:
        assert w.H % w.kv_heads == 0, w.name
        assert w.kind in ("forward", "train", "decode"), w.name
        if w.window:
            assert w.causal and 0 < w.window < w.N, w.name
        if w.uniform_head is not None:
            assert 0 <= w.uniform_head < w.H, w.name
        if w.dtype != torch.float32:
            assert w.d == 128, w.name


@pytest.mark.parametrize("w", [inputs.TINY_FP32], ids=lambda w: w.name)
def test_workload_inputs_match_the_recipe(w):
    a = inputs.workload_inputs(w, "cpu")
    b = inputs.attention_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, "cpu")
    assert all(torch.equal(x, y) for x, y in zip(a, b))
