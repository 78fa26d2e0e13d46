"""Plain, slow, fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
table or constant with the CUDA library in ``exact_attention_84_gb300/csrc``.

What it computes (sources are the four pages on FlashAttention; each
function cites the passage it follows):

* ``attention_forward``  -- the naive three-step definition
  S = Q.K^T * scale, P = row-softmax(S) with the row maximum subtracted,
  O = P.V, plus LSE = m + ln(l) per row.
  ("03. FlashAttention", section "Le probleme", steps 1-3;
  "FlashAttention ontleed", section "Het fysieke knelpunt"; the stored
  statistic m, l from "Geheugencomplexiteit: van O(N^2) naar O(N)".)
  FlashAttention is exact ("03. FlashAttention", "Benefices": "Exact";
  Lensa ML "FlashAttention", step 6), so its oracle is this definition.
* ``attention_backward`` -- the analytic gradient of O = softmax(S).V,
  which the pages leave to "recompute P from the stored statistics"
  ("03. FlashAttention", "Backward pass").  Written out by softmax
  calculus: D_i = sum_k dO_ik O_ik, dV = P^T dO, dP = dO V^T,
  dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.
* ``attention_decode`` -- one query row per (batch, head) over the whole
  KV cache, no mask ("FlashAttention ontleed", "Interactie met de
  KV-cache"; Lensa ML FAQ on decoding).  It does NOT split the cache:
  split-invariance is what the GPU path has to show.
* ``online_softmax_stats`` -- the running-max / running-sum update rule of
  Lensa ML "FlashAttention", step 4 "Online Softmax", used only to pin the
  definition against that page's worked example.
* ``tile_merged_attention_row`` -- one row computed as independent tile
  partials (o_t, lse_t) merged by their log-sum-exp weights, used only to
  pin the exactness claim of Lensa ML "FlashAttention", step 6.

Readings taken where the pages are silent:
* causal masking means key j is hidden from query i when j > i (square,
  top-left aligned);
* the stored statistic is one fp32 LSE = m + ln l in the natural log;
* a row whose every score is masked does not occur under the square causal
  mask (key 0 is always visible), so no special case is needed here.

Every function takes numpy arrays of any float dtype and computes in
float64.  Pins: tests/test_oracle.py.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attention_forward_gqa",
    "attention_backward_gqa",
    "attention_decode_gqa",
    "attention_forward",
    "attention_forward_rows",
    "attention_backward",
    "attention_decode",
    "online_softmax_stats",
    "tile_merged_attention_row",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _head_forward(q, k, v, scale, causal, rows, window=None, slope=None):
    """One head: q [Nq, d] (the query rows listed in ``rows``), k/v [Nk, d].

    Step 1 of "Le probleme": S = Q.K^T (times scale, "FlashAttention
    ontleed" pseudocode step 1 divides by sqrt(d)).  Step 2: the row softmax
    with its maximum subtracted before exponentiation (Lensa ML step 4:
    subtracting the maximum keeps the exponents small).  Step 3: O = P.V.
    """
    s = (q @ k.T) * scale                      # [Nq, Nk]
    if slope is not None:
        # ALiBi: linear bias -slope * |i - j| on the scaled score
        dist = np.abs(np.asarray(rows)[:, None] - np.arange(k.shape[0])[None, :])
        s = s - slope * dist
    if causal:
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > np.asarray(rows)[:, None], -np.inf, s)
    if window is not None:
        # sliding window: query i sees keys i - window + 1 .. i
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols < np.asarray(rows)[:, None] - window + 1, -np.inf, s)
    m = s.max(axis=1)                          # row maximum
    e = np.exp(s - m[:, None])                 # exp(-inf) = 0 for masked keys
    l = e.sum(axis=1)                          # row sum of exponentials
    p = e / l[:, None]                         # P = softmax(S)
    o = p @ v
    lse = m + np.log(l)
    return o, lse, p


def attention_forward(q, k, v, scale: float, causal: bool):
    """O = softmax(Q.K^T*scale [+ causal mask]).V and LSE for [..., N, d].

    Leading dimensions (batch, heads) are looped over one head at a time.
    Returns (O [..., N, d] float64, LSE [..., N] float64).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    lead = q.shape[:-2]
    n = q.shape[-2]
    o = np.empty(q.shape[:-1] + (v.shape[-1],), dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    rows = np.arange(n)
    for idx in np.ndindex(*lead):
        o[idx], lse[idx], _ = _head_forward(q[idx], k[idx], v[idx], scale, causal, rows)
    return o, lse


def attention_forward_rows(q_rows, k, v, rows, scale: float, causal: bool, window=None,
                           slope=None):
    """The same definition for a chosen subset of query rows of ONE head.

    ``q_rows`` [R, d] are the query vectors at positions ``rows`` (needed for
    the causal mask); ``k``, ``v`` [N, d] are the head's full key/value
    matrices.  Each output row depends only on its own query row, so this is
    the definition evaluated row by row, not a blocking of it.  ``window``
    and ``slope`` (optional) apply the sliding-window mask and the ALiBi
    bias described further down.
    """
    o, lse, _ = _head_forward(_f64(q_rows), _f64(k), _f64(v), scale, causal,
                              np.asarray(rows), window, slope)
    return o, lse


def attention_backward(q, k, v, do, scale: float, causal: bool, o=None):
    """Analytic gradients (dQ, dK, dV) of O = softmax(Q.K^T*scale).V.

    P is recomputed from Q and K ("03. FlashAttention", "Backward pass":
    only O and the softmax statistics are kept; P is recomputed).  Then, by
    the chain rule through the row softmax:
      dV = P^T dO
      dP = dO V^T
      D_i = sum_j P_ij dP_ij = sum_k dO_ik O_ik
      dS = P * (dP - D)          (softmax Jacobian applied row by row)
      dQ = scale * dS K,  dK = scale * dS^T Q
    ``o`` (optional): the forward output as stored (e.g. rounded to bf16);
    the backward keeps O from the forward pass, so D is formed from it.  By
    default the exact O of the definition is used.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    o_stored = None if o is None else _f64(o)
    lead = q.shape[:-2]
    n = q.shape[-2]
    rows = np.arange(n)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for idx in np.ndindex(*lead):
        o, _, p = _head_forward(q[idx], k[idx], v[idx], scale, causal, rows)
        if o_stored is not None:
            o = o_stored[idx]
        g = do[idx]
        dv[idx] = p.T @ g
        dp = g @ v[idx].T
        d_row = (g * o).sum(axis=1)
        ds = p * (dp - d_row[:, None])
        dq[idx] = scale * (ds @ k[idx])
        dk[idx] = scale * (ds.T @ q[idx])
    return dq, dk, dv


def attention_decode(q, kcache, vcache, scale: float):
    """One query token per (batch, head) against its whole KV cache.

    q [..., d], kcache/vcache [..., L, d].  No mask: the new token sees every
    cached position.  Returns (o [..., d], lse [...]).
    """
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    lead = q.shape[:-1]
    o = np.empty(lead + (vc.shape[-1],), dtype=np.float64)
    lse = np.empty(lead, dtype=np.float64)
    for idx in np.ndindex(*lead):
        s = (kc[idx] @ q[idx]) * scale         # [L]
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        o[idx] = (e @ vc[idx]) / l
        lse[idx] = m + math.log(l)
    return o, lse


def online_softmax_stats(x, chunk: int):
    """The pages' one-pass normaliser over a row of scores, chunk by chunk.

    Lensa ML "FlashAttention", step 4: m_new = max(m, chunk max) and
    l_new = l * e^(m - m_new) + sum e^(x - m_new), starting from m = -inf,
    l = 0.  Returns the list of (m, l) after each chunk.
    """
    x = _f64(x)
    m, l = -math.inf, 0.0
    trace = []
    for start in range(0, x.shape[0], chunk):
        c = x[start:start + chunk]
        m_new = max(m, float(c.max()))
        l = l * math.exp(m - m_new) + float(np.exp(c - m_new).sum())
        m = m_new
        trace.append((m, l))
    return trace


def tile_merged_attention_row(q, k, v, scale: float, tile: int):
    """One query row (no mask) computed tile by tile, then merged.

    Every tile of at most ``tile`` keys is treated as a small attention
    problem of its own: its scores, its own maximum and sum, its normalised
    output o_t and its log-sum-exp lse_t.  The row over all keys then
    follows from the partials alone: with L = ln sum_t e^(lse_t), a key of
    tile t carries weight e^(lse_t - L) times its weight inside the tile, so
    O = sum_t e^(lse_t - L) o_t and LSE = L.  This is the rescaling behind
    the running maximum and sum of Lensa ML "FlashAttention", step 4,
    applied across tiles; it is used only to pin the exactness claim of
    step 6 (tiled equals standard up to rounding).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    partials = []
    for start in range(0, k.shape[0], tile):
        kt, vt = k[start:start + tile], v[start:start + tile]
        s_t = (kt @ q) * scale
        m_t = float(s_t.max())
        e_t = np.exp(s_t - m_t)
        l_t = float(e_t.sum())
        partials.append(((e_t @ vt) / l_t, m_t + math.log(l_t)))
    lses = [lse_t for _, lse_t in partials]
    top = max(lses)
    total = top + math.log(math.fsum(math.exp(x - top) for x in lses))
    o = np.zeros(v.shape[-1], dtype=np.float64)
    for o_t, lse_t in partials:
        w = math.exp(lse_t - total)
        o = o + w * o_t
    return o, total


# --------------------------------------------------------------------------
# Grouped query heads and a causal sliding window.
#
# Grouped-query attention ("FlashAttention ontleed", "Interactie met de
# KV-cache": several query heads share the same key and value heads): with
# Hq query heads and Hkv key/value heads, query head h reads key/value head
# h // (Hq / Hkv).  Sliding window ("03. FlashAttention", "Variantes et
# extensions": only the K_j inside the window are considered): query i sees
# keys i - window + 1 .. i (used together with the causal mask).
# ALiBi ("03. FlashAttention", "Variantes et extensions": the linear bias
# integrated into the kernel): head h adds -slope_h * |i - j| to the scaled
# score S_ij = scale q_i.k_j before the softmax (under the causal mask this
# is slope_h * (j - i)); slopes are given per query head.
# --------------------------------------------------------------------------
def _kv_head(h, hq, hkv):
    return h // (hq // hkv)


def _slope(alibi_slopes, h):
    return None if alibi_slopes is None else float(alibi_slopes[h])


def attention_forward_gqa(q, k, v, scale: float, causal: bool, window=None, alibi_slopes=None):
    """q [B, Hq, N, d], k/v [B, Hkv, N, d] -> (O [B, Hq, N, d], LSE [B, Hq, N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, hq, n, _ = q.shape
    hkv = k.shape[1]
    o = np.empty(q.shape[:-1] + (v.shape[-1],), dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    rows = np.arange(n)
    for b in range(B):
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            o[b, h], lse[b, h], _ = _head_forward(q[b, h], k[b, g], v[b, g], scale, causal, rows,
                                                  window, _slope(alibi_slopes, h))
    return o, lse


def attention_backward_gqa(q, k, v, do, scale: float, causal: bool, window=None,
                           alibi_slopes=None, o=None):
    """Gradients for grouped heads: dQ per query head; dK, dV of a key/value
    head are the sums over the query heads that read it.  ``o``: the stored
    forward output, as in ``attention_backward``."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    o_given = None if o is None else _f64(o)
    B, hq, n, _ = q.shape
    hkv = k.shape[1]
    rows = np.arange(n)
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            o, _, p = _head_forward(q[b, h], k[b, g], v[b, g], scale, causal, rows, window,
                                    _slope(alibi_slopes, h))
            if o_given is not None:
                o = o_given[b, h]
            gr = do[b, h]
            dv[b, g] += p.T @ gr                  # dV summed over the group
            dpg = gr @ v[b, g].T
            dsum = (gr * o).sum(axis=1)           # D_i = dO_i . O_i
            dsg = p * (dpg - dsum[:, None])
            dq[b, h] = scale * (dsg @ k[b, g])
            dk[b, g] += scale * (dsg.T @ q[b, h])  # dK summed over the group
    return dq, dk, dv


def attention_decode_gqa(q, kcache, vcache, scale: float, alibi_slopes=None):
    """q [B, Hq, d], caches [B, Hkv, L, d] -> (o [B, Hq, d], lse [B, Hq]).
    The new query sits at position L - 1, after every cached row (ALiBi
    distance L - 1 - j)."""
    q, kc, vc = _f64(q), _f64(kcache), _f64(vcache)
    B, hq, _ = q.shape
    hkv = kc.shape[1]
    o = np.empty(q.shape[:-1] + (vc.shape[-1],), dtype=np.float64)
    lse = np.empty((B, hq), dtype=np.float64)
    for b in range(B):
        for h in range(hq):
            g = _kv_head(h, hq, hkv)
            s = (kc[b, g] @ q[b, h]) * scale
            if alibi_slopes is not None:
                s = s - float(alibi_slopes[h]) * (s.shape[0] - 1 - np.arange(s.shape[0]))
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            o[b, h] = (e @ vc[b, g]) / l
            lse[b, h] = m + math.log(l)
    return o, lse
