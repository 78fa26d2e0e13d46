"""FLOP and byte accounting used by the bench's throughput and roofline
figures (host arithmetic only).

Conventions: the forward pass counts the two matrix products, 2 N^2 d
multiply-adds each, i.e. 4 B H N^2 d FLOPs, halved under the causal mask; the
backward pass counts 2.5 times the forward (five products instead of two).
Decode is bound by reading the KV cache once.

The page figures these reproduce (Lensa ML "FlashAttention", steps 2 and 5)
are pinned in tests/test_accounting.py.
"""

from __future__ import annotations


def forward_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def backward_flops(B, H, N, d, causal):
    return 2.5 * forward_flops(B, H, N, d, causal)


def visible_pairs(N, causal, window=0):
    """Number of (query, key) pairs the mask leaves visible in one head: the
    exact count N^2, N(N+1)/2 (causal), or sum_i min(i+1, w) (window w)."""
    if window and causal and window < N:
        return window * (window + 1) // 2 + (N - window) * window
    return N * (N + 1) // 2 if causal else N * N


def masked_forward_flops(B, H, N, d, causal, window=0):
    """4 d FLOPs per visible (query, key) pair and query head.  Only the
    windowed workloads use it: the plain forward keeps the N^2 / 2 causal
    convention above."""
    return 4.0 * B * H * d * visible_pairs(N, causal, window)


def forward_min_bytes(B, H, N, d, elem=2):
    """Q, K, V read once, O written once, fp32 LSE written once."""
    return 4 * B * H * N * d * elem + 4 * B * H * N


def backward_min_bytes(B, H, N, d, elem=2):
    """Q, K, V, O, dO read; dQ, dK, dV written; LSE read (D computed)."""
    return 8 * B * H * N * d * elem + 4 * B * H * N


def decode_kv_bytes(B, H, L, d, elem=2):
    """The KV cache read once: the algorithmic traffic of one decode call
    (H = key/value heads: with grouped query heads the cache has Hkv)."""
    return 2 * B * H * L * d * elem


def decode_min_bytes(B, H, L, d, elem=2):
    """KV cache plus the query and output vectors."""
    return decode_kv_bytes(B, H, L, d, elem) + 2 * B * H * d * elem


def standard_attention_hbm_elements(N, d):
    """Naive three-kernel attention, one head: Q, K, V read, S written and read,
    P written and read, O written -- about 4 N^2 + 4 N d elements."""
    return 4 * N * N + 4 * N * d


def standard_hbm_accesses(N, d):
    """Theta(N d + N^2) HBM accesses of standard attention (constant 1)."""
    return N * d + N * N


def flash_hbm_accesses(N, d, M):
    """Theta(N^2 d^2 / M) HBM accesses of the tiled kernel (constant 1),
    M = on-chip memory in elements."""
    return N * N * d * d / M
