"""Pins that tie the fp64 oracle to facts fixed outside itself.

Each ``pin_*`` takes an oracle module (the real ``oracle.attention``, or a
copy with a planted mistake) and raises AssertionError when the oracle
disagrees with what the pages print or what the mathematics forces.  The
checks never re-type the oracle's own formula: they use values printed on
the pages, closed forms, invariances, brute-force scalar loops, finite
differences and PyTorch's own fp64 CPU attention as a library special case.
"""

from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition("=")
            nums = [float(t) for t in rest.split()]
            vals[key.strip()] = nums if len(nums) > 1 else nums[0]
    return vals


def _rng(seed):
    return np.random.default_rng(seed)


# --- brute force: scalar loops over the definition, math.exp and fsum ------
def brute_forward(q, k, v, scale, causal):
    n, d = len(q), len(q[0])
    nk = len(k)
    o = [[0.0] * len(v[0]) for _ in range(n)]
    lse = [0.0] * n
    for i in range(n):
        scores = []
        for j in range(nk):
            if causal and j > i:
                continue
            scores.append((j, scale * math.fsum(q[i][t] * k[j][t] for t in range(d))))
        top = max(s for _, s in scores)
        w = [(j, math.exp(s - top)) for j, s in scores]
        tot = math.fsum(x for _, x in w)
        for c in range(len(v[0])):
            o[i][c] = math.fsum(x * v[j][c] for j, x in w) / tot
        lse[i] = top + math.log(tot)
    return np.array(o), np.array(lse)


def _scalar_loss(orc, q, k, v, do, scale, causal):
    o, _ = orc.attention_forward(q, k, v, scale, causal)
    return float((o * do).sum())


# --- pins -------------------------------------------------------------------
def pin_walkthrough_softmax(orc):
    """Lensa ML step 4: the printed full softmax of the eight scores."""
    g = read_golden("online_softmax_walkthrough.txt")
    x = np.array(g["scores"])
    n = x.size
    # One query of width 1 equal to 1, keys equal to the scores, scale 1 and
    # V = identity: row 0 of O is then softmax(x) itself.
    q = np.ones((1, 1, n, 1))
    k = x.reshape(1, 1, n, 1)
    v = np.eye(n).reshape(1, 1, n, n)
    o, lse = orc.attention_forward(q, k, v, 1.0, False)
    printed = np.array(g["softmax_2dp"])
    assert np.all(np.abs(o[0, 0, 0] - printed) <= 0.005 + 1e-12), o[0, 0, 0]
    assert abs(o[0, 0, 0].sum() - 1.0) < 1e-14
    want_lse = math.log(math.fsum(math.exp(t) for t in x))
    assert abs(lse[0, 0, 0] - want_lse) < 1e-13
    # The same scores through the decode path (one query over a cache).
    od, lsed = orc.attention_decode(np.ones((1, 1)), x.reshape(1, n, 1),
                                    np.eye(n).reshape(1, n, n), 1.0)
    assert np.all(np.abs(od[0] - printed) <= 0.005 + 1e-12), od[0]
    assert abs(lsed[0] - want_lse) < 1e-13


def pin_walkthrough_online(orc):
    """Lensa ML step 4: 4 chunks of 2; the running (m, l) after the last chunk
    gives the same normaliser as the full softmax for any chunk size."""
    g = read_golden("online_softmax_walkthrough.txt")
    x = np.array(g["scores"])
    trace = orc.online_softmax_stats(x, int(g["chunk_size"]))
    assert len(trace) == int(g["num_chunks"])
    full = math.fsum(math.exp(t) for t in x)
    finals = []
    for chunk in (1, 2, 4, 8):
        m, l = orc.online_softmax_stats(x, chunk)[-1]
        assert m == max(x) == 4.5
        finals.append(m + math.log(l))
    for f in finals:
        assert abs(f - math.log(full)) < 1e-14
    # After chunk 2 the maximum is x2 = 3.0; chunk 3 holds x5 = 4.5, so the
    # old sum is rescaled by e^(3.0 - 4.5) before the new terms are added.
    (m2, l2), (m3, l3) = trace[1], trace[2]
    assert m2 == 3.0 and m3 == 4.5
    want_l3 = l2 * math.exp(3.0 - 4.5) + math.exp(4.5 - 4.5) + math.exp(1.8 - 4.5)
    assert abs(l3 - want_l3) < 1e-14
    want_l2 = math.fsum(math.exp(t - 3.0) for t in x[:4])
    assert abs(l2 - want_l2) < 1e-14


def pin_exactness(orc):
    """Lensa ML step 6: one query, d = 8, 4 tiles of at most 4 keys; tiled and
    standard agree to rounding (the page prints 2.2e-16)."""
    g = read_golden("exactness_check.txt")
    d = int(g["head_dim"])
    n = int(g["tiles"] * g["keys_per_tile"])
    worst = 0.0
    for seed in range(20):
        r = _rng(seed)
        q = r.standard_normal((1, d))
        k = r.standard_normal((n, d))
        v = r.standard_normal((n, d))
        scale = 1 / math.sqrt(d)
        o_std, lse_std = orc.attention_forward(q[None, None], k[None, None], v[None, None],
                                               scale, False)
        o_t, lse_t = orc.tile_merged_attention_row(q[0], k, v, scale, int(g["keys_per_tile"]))
        worst = max(worst, float(np.abs(o_std[0, 0, 0] - o_t).max()),
                    abs(float(lse_std[0, 0, 0]) - lse_t))
    assert worst <= 5 * g["max_abs_diff_printed"] + 1e-16, worst


def pin_brute_force(orc):
    """Scalar loops with math.exp / math.fsum on tiny shapes."""
    for seed in range(6):
        r = _rng(100 + seed)
        n, d, dv = 1 + seed, 2 + seed % 3, 1 + (seed * 2) % 5
        q = r.standard_normal((n, d))
        k = r.standard_normal((n, d))
        v = r.standard_normal((n, dv))
        scale = 0.3 + 0.1 * seed
        for causal in (False, True):
            o, lse = orc.attention_forward(q[None], k[None], v[None], scale, causal)
            bo, blse = brute_forward(q.tolist(), k.tolist(), v.tolist(), scale, causal)
            assert np.abs(o[0] - bo).max() < 1e-13
            assert np.abs(lse[0] - blse).max() < 1e-13
    # Non-square (more keys than queries) and decode against the same loops.
    r = _rng(7)
    q = r.standard_normal((3, 4))
    k = r.standard_normal((9, 4))
    v = r.standard_normal((9, 5))
    od, lsed = orc.attention_decode(q, np.stack([k] * 3), np.stack([v] * 3), 0.7)
    bo, blse = brute_forward(q.tolist(), k.tolist(), v.tolist(), 0.7, False)
    assert np.abs(od - bo).max() < 1e-13 and np.abs(lsed - blse).max() < 1e-13


def pin_uniform_keys(orc):
    """All keys identical: every visible key gets the same weight."""
    r = _rng(11)
    n, d = 12, 6
    q = r.standard_normal((n, d))
    k = np.tile(r.standard_normal((1, d)), (n, 1))
    v = r.standard_normal((n, d))
    scale = 1 / math.sqrt(d)
    o, lse = orc.attention_forward(q[None], k[None], v[None], scale, False)
    assert np.abs(o[0] - v.mean(axis=0)[None]).max() < 1e-13
    assert np.abs(lse[0] - (scale * q @ k[0] + math.log(n))).max() < 1e-13
    o, lse = orc.attention_forward(q[None], k[None], v[None], scale, True)
    for i in range(n):
        assert np.abs(o[0, i] - v[: i + 1].mean(axis=0)).max() < 1e-13
        assert abs(lse[0, i] - (scale * q[i] @ k[0] + math.log(i + 1))) < 1e-13
    # scale = 0 makes every score equal as well.
    k2 = r.standard_normal((n, d))
    o, lse = orc.attention_forward(q[None], k2[None], v[None], 0.0, False)
    assert np.abs(o[0] - v.mean(axis=0)[None]).max() < 1e-13
    assert np.abs(lse[0] - math.log(n)).max() < 1e-13


def pin_causal_row0(orc):
    """Under the causal mask query 0 sees key 0 only; the last query sees all."""
    r = _rng(12)
    n, d = 9, 5
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    o, lse = orc.attention_forward(q[None], k[None], v[None], 0.5, True)
    assert np.abs(o[0, 0] - v[0]).max() < 1e-14
    assert abs(lse[0, 0] - 0.5 * q[0] @ k[0]) < 1e-14
    of, lsef = orc.attention_forward(q[None], k[None], v[None], 0.5, False)
    assert np.abs(o[0, -1] - of[0, -1]).max() < 1e-14
    assert abs(lse[0, -1] - lsef[0, -1]) < 1e-14
    assert np.abs(o[0, 1] - of[0, 1]).max() > 1e-6   # row 1 does differ


def pin_invariances(orc):
    """V = 1 gives O = 1; shifting every key by c shifts LSE by scale q.c and
    leaves O alone; permuting the keys (no mask) changes nothing; a constant
    added to every score (large enough to overflow e^x in fp64) changes
    nothing either."""
    r = _rng(13)
    n, d = 10, 4
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    s = 0.6
    o1, _ = orc.attention_forward(q[None], k[None], np.ones((1, n, 3)), s, True)
    assert np.abs(o1 - 1).max() < 1e-14
    c = r.standard_normal(d)
    for causal in (False, True):
        o, lse = orc.attention_forward(q[None], k[None], v[None], s, causal)
        o2, lse2 = orc.attention_forward(q[None], (k + c)[None], v[None], s, causal)
        assert np.abs(o - o2).max() < 1e-12
        assert np.abs(lse2[0] - lse[0] - s * q @ c).max() < 1e-12
    perm = r.permutation(n)
    o, lse = orc.attention_forward(q[None], k[None], v[None], s, False)
    o3, lse3 = orc.attention_forward(q[None], k[perm][None], v[perm][None], s, False)
    assert np.abs(o - o3).max() < 1e-13 and np.abs(lse - lse3).max() < 1e-13
    # e^800 overflows fp64: only a max-subtracted softmax survives this.
    g = read_golden("online_softmax_walkthrough.txt")
    x = np.array(g["scores"])
    m = x.size
    v8 = np.eye(m).reshape(1, m, m)
    base, lb = orc.attention_forward(np.ones((1, 1, 1)), x.reshape(1, m, 1), v8, 1.0, False)
    big, lbig = orc.attention_forward(np.ones((1, 1, 1)), (x + 800).reshape(1, m, 1), v8, 1.0,
                                      False)
    assert np.all(np.isfinite(big)) and np.abs(big - base).max() < 1e-13
    assert abs(lbig[0, 0] - lb[0, 0] - 800) < 1e-10
    od, ld = orc.attention_decode(np.ones((1, 1)), (x + 800).reshape(1, m, 1), v8, 1.0)
    assert np.all(np.isfinite(od)) and np.abs(od - base[0]).max() < 1e-13


def pin_backward_finite_diff(orc):
    """Central differences of L = sum(O * dO) in fp64 on tiny shapes."""
    for causal in (False, True):
        r = _rng(21 + causal)
        n, d = 5, 3
        q, k, v, do = (r.standard_normal((1, n, d)) for _ in range(4))
        s = 0.8
        dq, dk, dv = orc.attention_backward(q, k, v, do, s, causal)
        h = 1e-6
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v, name: xp}
                args_m = {"q": q, "k": k, "v": v, name: xm}
                lp = _scalar_loss(orc, args_p["q"], args_p["k"], args_p["v"], do, s, causal)
                lm = _scalar_loss(orc, args_m["q"], args_m["k"], args_m["v"], do, s, causal)
                num[idx] = (lp - lm) / (2 * h)
            err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
            assert err < 1e-6, (name, causal, err)


def pin_backward_identities(orc):
    """Rows of P sum to one, so sum_j dV_j = sum_i dO_i; rows of dS sum to
    zero, so sum_j dK_j = 0."""
    r = _rng(31)
    q, k, v, do = (r.standard_normal((2, 7, 4)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.attention_backward(q, k, v, do, 0.5, causal)
        assert np.abs(dv.sum(axis=-2) - do.sum(axis=-2)).max() < 1e-12
        assert np.abs(dk.sum(axis=-2)).max() < 1e-12


def pin_backward_stored_o(orc):
    """The backward forms D from the O it is given: with the exact O nothing
    changes; shifting row i of O by c changes D_i by c * sum_k dO_ik, which
    moves dQ_i by -scale * dD_i * (P K)_i and dK_j by -scale * sum_i P_ij
    dD_i Q_i and leaves dV alone."""
    r = _rng(71)
    n, d = 6, 4
    q, k, v, do = (r.standard_normal((1, n, d)) for _ in range(4))
    o, lse = orc.attention_forward(q, k, v, 0.5, True)
    base = orc.attention_backward(q, k, v, do, 0.5, True)
    same = orc.attention_backward(q, k, v, do, 0.5, True, o=o)
    for a, b in zip(base, same):
        assert np.abs(a - b).max() < 1e-15
    shift = np.zeros((1, n, 1))
    shift[0, 2, 0], shift[0, 4, 0] = 0.3, -0.7
    moved = orc.attention_backward(q, k, v, do, 0.5, True, o=o + shift)
    dd = shift[0, :, 0] * do[0].sum(axis=1)                       # change of D_i
    s = 0.5 * q[0] @ k[0].T
    s = np.where(np.arange(n)[None, :] > np.arange(n)[:, None], -np.inf, s)
    p = np.exp(s - lse[0][:, None])
    want_dq = base[0][0] - 0.5 * dd[:, None] * (p @ k[0])
    want_dk = base[1][0] - 0.5 * (p * dd[:, None]).T @ q[0]
    assert np.abs(moved[0][0] - want_dq).max() < 1e-13
    assert np.abs(moved[1][0] - want_dk).max() < 1e-13
    assert np.abs(moved[2] - base[2]).max() < 1e-15
    g = orc.attention_backward_gqa(q[None], k[None], v[None], do[None], 0.5, True, o=(o + shift)[None])
    for a, b in zip(g, moved):
        assert np.abs(a[0] - b).max() < 1e-14


def pin_torch_sdpa(orc):
    """Library special case: PyTorch's fp64 CPU attention and autograd."""
    import torch
    import torch.nn.functional as F

    g = torch.Generator().manual_seed(5)
    for causal in (False, True):
        q, k, v, do = (torch.randn(2, 3, 33, 16, generator=g, dtype=torch.float64)
                       for _ in range(4))
        scale = 1 / math.sqrt(16)
        qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
        ref = F.scaled_dot_product_attention(qq, kk, vv, is_causal=causal, scale=scale)
        ref.backward(do)
        o, lse = orc.attention_forward(q.numpy(), k.numpy(), v.numpy(), scale, causal)
        assert np.abs(o - ref.detach().numpy()).max() < 1e-12
        s = (q @ k.transpose(-1, -2)) * scale
        if causal:
            s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), float("-inf"))
        assert np.abs(lse - torch.logsumexp(s, dim=-1).numpy()).max() < 1e-12
        dq, dk, dv = orc.attention_backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(),
                                            scale, causal)
        assert np.abs(dq - qq.grad.numpy()).max() < 1e-12
        assert np.abs(dk - kk.grad.numpy()).max() < 1e-12
        assert np.abs(dv - vv.grad.numpy()).max() < 1e-12
    q1 = torch.randn(4, 2, 1, 8, generator=g, dtype=torch.float64)
    kc = torch.randn(4, 2, 50, 8, generator=g, dtype=torch.float64)
    vc = torch.randn(4, 2, 50, 8, generator=g, dtype=torch.float64)
    ref = F.scaled_dot_product_attention(q1, kc, vc, scale=0.25)
    od, lsed = orc.attention_decode(q1[:, :, 0].numpy(), kc.numpy(), vc.numpy(), 0.25)
    assert np.abs(od - ref[:, :, 0].numpy()).max() < 1e-12
    s = (q1 @ kc.transpose(-1, -2))[:, :, 0] * 0.25
    assert np.abs(lsed - torch.logsumexp(s, dim=-1).numpy()).max() < 1e-12


def pin_rows_subset(orc):
    """Row subsets give the rows of the full result (used at large sizes)."""
    r = _rng(41)
    n, d = 20, 4
    q, k, v = (r.standard_normal((n, d)) for _ in range(3))
    rows = np.array([0, 3, 19, 7])
    for causal in (False, True):
        of, lf = orc.attention_forward(q[None], k[None], v[None], 0.5, causal)
        orow, lrow = orc.attention_forward_rows(q[rows], k, v, rows, 0.5, causal)
        assert np.abs(orow - of[0, rows]).max() < 1e-14
        assert np.abs(lrow - lf[0, rows]).max() < 1e-14
    # Row i of a causal result equals the non-causal result over keys 0..i.
    i = 6
    oc, lc = orc.attention_forward_rows(q[[i]], k, v, [i], 0.5, True)
    on, ln = orc.attention_forward_rows(q[[i]], k[: i + 1], v[: i + 1], [i], 0.5, False)
    assert np.abs(oc - on).max() < 1e-14 and np.abs(lc - ln).max() < 1e-14


def brute_forward_window(q, k, v, scale, window):
    """Scalar loop: causal attention of row i over keys max(0, i-window+1)..i."""
    n = len(q)
    o = np.zeros((n, len(v[0])))
    lse = np.zeros(n)
    for i in range(n):
        js = range(max(0, i - window + 1), i + 1)
        sc = {j: scale * math.fsum(q[i][t] * k[j][t] for t in range(len(q[0]))) for j in js}
        top = max(sc.values())
        w = {j: math.exp(x - top) for j, x in sc.items()}
        tot = math.fsum(w.values())
        for c in range(len(v[0])):
            o[i, c] = math.fsum(w[j] * v[j][c] for j in js) / tot
        lse[i] = top + math.log(tot)
    return o, lse


def pin_gqa_repeat_kv(orc):
    """Grouped heads are ordinary heads over repeated K/V: query head h reads
    key/value head h // (Hq/Hkv), so the grouped result equals the pinned
    per-head definition on K/V repeated group-wise, and the grouped dK, dV are
    the per-head gradients summed over each group."""
    r = _rng(51)
    b, hq, hkv, n, d = 2, 6, 2, 9, 4
    q, do = (r.standard_normal((b, hq, n, d)) for _ in range(2))
    k, v = (r.standard_normal((b, hkv, n, d)) for _ in range(2))
    grp = hq // hkv
    kr, vr = np.repeat(k, grp, axis=1), np.repeat(v, grp, axis=1)
    for causal in (False, True):
        o, lse = orc.attention_forward_gqa(q, k, v, 0.5, causal)
        om, lm = orc.attention_forward(q, kr, vr, 0.5, causal)
        assert np.abs(o - om).max() < 1e-14 and np.abs(lse - lm).max() < 1e-14
        dq, dk, dv = orc.attention_backward_gqa(q, k, v, do, 0.5, causal)
        dqm, dkm, dvm = orc.attention_backward(q, kr, vr, do, 0.5, causal)
        assert np.abs(dq - dqm).max() < 1e-13
        assert np.abs(dk - dkm.reshape(b, hkv, grp, n, d).sum(axis=2)).max() < 1e-13
        assert np.abs(dv - dvm.reshape(b, hkv, grp, n, d).sum(axis=2)).max() < 1e-13
    # one group (Hkv = Hq) is the per-head definition itself
    o1, l1 = orc.attention_forward_gqa(q, q, do, 0.5, True)
    om1, lm1 = orc.attention_forward(q, q, do, 0.5, True)
    assert np.abs(o1 - om1).max() < 1e-15 and np.abs(l1 - lm1).max() < 1e-15
    qd = r.standard_normal((b, hq, d))
    kc, vc = (r.standard_normal((b, hkv, 13, d)) for _ in range(2))
    od, ld = orc.attention_decode_gqa(qd, kc, vc, 0.5)
    odm, ldm = orc.attention_decode(qd, np.repeat(kc, grp, axis=1), np.repeat(vc, grp, axis=1),
                                    0.5)
    assert np.abs(od - odm).max() < 1e-14 and np.abs(ld - ldm).max() < 1e-14


def pin_window_closed_forms(orc):
    """Sliding window: width 1 leaves one key per row (O_i = V_i, LSE_i =
    scale q_i.k_i); width >= N is plain causal attention; otherwise a scalar
    loop over the window's keys."""
    r = _rng(53)
    n, d = 11, 3
    q, k, v, do = (r.standard_normal((1, 1, n, d)) for _ in range(4))
    o, lse = orc.attention_forward_gqa(q, k, v, 0.7, True, window=1)
    assert np.abs(o - v).max() < 1e-15
    assert np.abs(lse[0, 0] - 0.7 * (q[0, 0] * k[0, 0]).sum(axis=1)).max() < 1e-14
    dq, dk, dv = orc.attention_backward_gqa(q, k, v, do, 0.7, True, window=1)
    assert np.abs(dv - do).max() < 1e-15       # P = I
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    for w in (n, n + 5):
        ow, lw = orc.attention_forward_gqa(q, k, v, 0.7, True, window=w)
        oc, lc = orc.attention_forward(q, k, v, 0.7, True)
        assert np.abs(ow - oc).max() < 1e-15 and np.abs(lw - lc).max() < 1e-15
    for w in (2, 4, 7):
        ob, lb = brute_forward_window(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                                      0.7, w)
        ow, lw = orc.attention_forward_gqa(q, k, v, 0.7, True, window=w)
        assert np.abs(ow[0, 0] - ob).max() < 1e-13 and np.abs(lw[0, 0] - lb).max() < 1e-13
        rows = np.array([0, w - 1, w, n - 1])
        orow, lrow = orc.attention_forward_rows(q[0, 0, rows], k[0, 0], v[0, 0], rows, 0.7,
                                                True, window=w)
        assert np.abs(orow - ob[rows]).max() < 1e-13 and np.abs(lrow - lb[rows]).max() < 1e-13


def pin_gqa_window_torch(orc):
    """Library special case: PyTorch's fp64 attention with grouped heads and
    an explicit boolean window mask, and its autograd gradients."""
    import torch
    import torch.nn.functional as F

    g = torch.Generator().manual_seed(7)
    b, hq, hkv, n, d = 2, 4, 2, 37, 8
    q, do = (torch.randn(b, hq, n, d, generator=g, dtype=torch.float64) for _ in range(2))
    k, v = (torch.randn(b, hkv, n, d, generator=g, dtype=torch.float64) for _ in range(2))
    idx = torch.arange(n)
    for window in (None, 5, 16):
        allowed = idx[None, :] <= idx[:, None]
        if window is not None:
            allowed &= idx[None, :] > idx[:, None] - window
        qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=allowed, scale=0.3,
                                             enable_gqa=True)
        ref.backward(do)
        o, lse = orc.attention_forward_gqa(q.numpy(), k.numpy(), v.numpy(), 0.3, True, window)
        assert np.abs(o - ref.detach().numpy()).max() < 1e-12
        s = (q @ k.repeat_interleave(hq // hkv, dim=1).transpose(-1, -2)) * 0.3
        s = s.masked_fill(~allowed, float("-inf"))
        assert np.abs(lse - torch.logsumexp(s, dim=-1).numpy()).max() < 1e-12
        dq, dk, dv = orc.attention_backward_gqa(q.numpy(), k.numpy(), v.numpy(), do.numpy(),
                                                0.3, True, window)
        assert np.abs(dq - qq.grad.numpy()).max() < 1e-12
        assert np.abs(dk - kk.grad.numpy()).max() < 1e-12
        assert np.abs(dv - vv.grad.numpy()).max() < 1e-12
    q1 = torch.randn(3, 8, 1, 16, generator=g, dtype=torch.float64)
    kc, vc = (torch.randn(3, 2, 40, 16, generator=g, dtype=torch.float64) for _ in range(2))
    ref = F.scaled_dot_product_attention(q1, kc, vc, scale=0.25, enable_gqa=True)
    od, _ = orc.attention_decode_gqa(q1[:, :, 0].numpy(), kc.numpy(), vc.numpy(), 0.25)
    assert np.abs(od - ref[:, :, 0].numpy()).max() < 1e-12


def pin_alibi_closed_forms(orc):
    """ALiBi: identical keys leave only the bias, so causal row i weights key
    j by e^(-m (i - j)), a geometric series with a closed-form sum; slope 0
    is plain attention; a steep slope leaves only the diagonal."""
    r = _rng(61)
    n, d = 9, 4
    q, v = (r.standard_normal((1, 2, n, d)) for _ in range(2))
    k = np.repeat(r.standard_normal((1, 1, 1, d)), n, axis=2).repeat(2, axis=1)
    slopes = np.array([0.5, 0.125])
    o, lse = orc.attention_forward_gqa(q, k, v, 0.7, True, alibi_slopes=slopes)
    for h in range(2):
        m = slopes[h]
        for i in range(n):
            w = np.exp(-m * (i - np.arange(i + 1)))
            want = (w[:, None] * v[0, h, :i + 1]).sum(axis=0) / w.sum()
            assert np.abs(o[0, h, i] - want).max() < 1e-14
            series = (1 - math.exp(-m * (i + 1))) / (1 - math.exp(-m))
            assert abs(lse[0, h, i] - (0.7 * q[0, h, i] @ k[0, h, 0] + math.log(series))) < 1e-13
    # non-causal: the bias is symmetric in |i - j|
    o_nc, _ = orc.attention_forward_gqa(q, k, v, 0.7, False, alibi_slopes=slopes)
    for h in range(2):
        w = np.exp(-slopes[h] * np.abs(3 - np.arange(n)))
        want = (w[:, None] * v[0, h]).sum(axis=0) / w.sum()
        assert np.abs(o_nc[0, h, 3] - want).max() < 1e-14
    q2, k2, v2 = (r.standard_normal((1, 2, n, d)) for _ in range(3))
    o0, l0 = orc.attention_forward_gqa(q2, k2, v2, 0.5, True, alibi_slopes=np.zeros(2))
    ob, lb = orc.attention_forward(q2, k2, v2, 0.5, True)
    assert np.abs(o0 - ob).max() < 1e-15 and np.abs(l0 - lb).max() < 1e-15
    os_, ls = orc.attention_forward_gqa(q2, k2, v2, 0.5, False, alibi_slopes=np.full(2, 2000.0))
    assert np.abs(os_ - v2).max() < 1e-15
    assert np.abs(ls - 0.5 * (q2 * k2).sum(-1)).max() < 1e-12
    # decode: the new token is at position L - 1
    od, ld = orc.attention_decode_gqa(q2[:, :, -1], k2, v2, 0.5, alibi_slopes=slopes)
    of, lf = orc.attention_forward_gqa(q2, k2, v2, 0.5, True, alibi_slopes=slopes)
    assert np.abs(od - of[:, :, -1]).max() < 1e-14 and np.abs(ld - lf[:, :, -1]).max() < 1e-14


def pin_alibi_torch(orc):
    """Library special case: PyTorch's fp64 attention with the bias given as
    a float mask (-inf where causal hides a key), and its autograd gradients;
    grouped heads and a window on top."""
    import torch
    import torch.nn.functional as F

    g = torch.Generator().manual_seed(9)
    b, hq, hkv, n, d = 2, 4, 2, 29, 8
    q, do = (torch.randn(b, hq, n, d, generator=g, dtype=torch.float64) for _ in range(2))
    k, v = (torch.randn(b, hkv, n, d, generator=g, dtype=torch.float64) for _ in range(2))
    slopes = torch.tensor([0.5, 0.25, 0.125, 0.0625], dtype=torch.float64)
    idx = torch.arange(n)
    dist = (idx[:, None] - idx[None, :]).abs().to(torch.float64)
    for causal, window in ((False, None), (True, None), (True, 7)):
        bias = -slopes[:, None, None] * dist
        if causal:
            bias = bias.masked_fill(idx[None, :] > idx[:, None], float("-inf"))
        if window:
            bias = bias.masked_fill(idx[None, :] <= idx[:, None] - window, float("-inf"))
        qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=bias, scale=0.3,
                                             enable_gqa=True)
        ref.backward(do)
        o, lse = orc.attention_forward_gqa(q.numpy(), k.numpy(), v.numpy(), 0.3, causal, window,
                                           slopes.numpy())
        assert np.abs(o - ref.detach().numpy()).max() < 1e-12
        s = (q @ k.repeat_interleave(hq // hkv, dim=1).transpose(-1, -2)) * 0.3 + bias
        assert np.abs(lse - torch.logsumexp(s, dim=-1).numpy()).max() < 1e-12
        dq, dk, dv = orc.attention_backward_gqa(q.numpy(), k.numpy(), v.numpy(), do.numpy(),
                                                0.3, causal, window, slopes.numpy())
        assert np.abs(dq - qq.grad.numpy()).max() < 1e-12
        assert np.abs(dk - kk.grad.numpy()).max() < 1e-12
        assert np.abs(dv - vv.grad.numpy()).max() < 1e-12


ALL_PINS = [
    pin_walkthrough_softmax,
    pin_walkthrough_online,
    pin_exactness,
    pin_brute_force,
    pin_uniform_keys,
    pin_causal_row0,
    pin_invariances,
    pin_backward_finite_diff,
    pin_backward_identities,
    pin_backward_stored_o,
    pin_torch_sdpa,
    pin_rows_subset,
    pin_gqa_repeat_kv,
    pin_window_closed_forms,
    pin_gqa_window_torch,
    pin_alibi_closed_forms,
    pin_alibi_torch,
]
