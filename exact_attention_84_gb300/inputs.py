"""Seeded synthetic inputs shared by the tests, the bench and the oracle's
callers.  This module draws random numbers and nothing else: it holds none of
the attention arithmetic.

Recipe: one ``torch.Generator`` on the target device, seeded once per
workload; tensors are drawn in the order Q, K, V (, dO); each tensor is drawn
batch by batch as fp32 standard normals of shape [H, N, d] and then rounded
to the storage dtype (bf16: round to nearest even).  The oracle always reads
the very bytes the GPU reads, so parity does not depend on the generator.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int          # sequence length (KV length for decode)
    d: int
    dtype: torch.dtype
    seed: int
    causal: bool = False
    kind: str = "forward"        # forward | train | decode
    uniform_head: int | None = None   # head whose K rows all equal its row 0
    Hkv: int | None = None       # key/value heads (grouped query heads); None: H
    window: int = 0              # causal sliding window width; 0: none

    @property
    def kv_heads(self) -> int:
        return self.H if self.Hkv is None else self.Hkv


# The synthetic workloads, by what they are.
TINY_FP32 = Workload("tiny fp32 forward B1 H1 N256 d64", 1, 1, 256, 64, torch.float32, 0)
FWD_N2048 = Workload("bf16 forward B4 H16 N2048 d128", 4, 16, 2048, 128, torch.bfloat16, 1)
LONG_CAUSAL = Workload("bf16 causal forward B1 H32 N8192 d128", 1, 32, 8192, 128,
                       torch.bfloat16, 2, causal=True, uniform_head=31)
TRAIN_N4096 = Workload("bf16 causal forward+backward B8 H32 N4096 d128", 8, 32, 4096, 128,
                       torch.bfloat16, 3, causal=True, kind="train")
DECODE_L32K = Workload("bf16 split-KV decode B64 H32 Lkv32768 d128", 64, 32, 32768, 128,
                       torch.bfloat16, 4, kind="decode")
# Grouped query heads (4 query heads per key/value head) and a sliding window.
GQA_TRAIN_N4096 = Workload("bf16 causal GQA forward+backward B8 Hq32 Hkv8 N4096 d128", 8, 32,
                           4096, 128, torch.bfloat16, 5, causal=True, kind="train", Hkv=8)
WINDOW_N8192 = Workload("bf16 causal sliding-window (w=1024) forward B1 H32 N8192 d128", 1, 32,
                        8192, 128, torch.bfloat16, 6, causal=True, window=1024)
GQA_DECODE_L32K = Workload("bf16 GQA split-KV decode B64 Hq32 Hkv8 Lkv32768 d128", 64, 32,
                           32768, 128, torch.bfloat16, 7, kind="decode", Hkv=8)
# FP8 (E4M3) inputs: N(0,1) draws times FP8_AMP, rounded to E4M3; descale
# factor 1/FP8_AMP for each tensor.
FP8_LONG_CAUSAL = Workload("fp8 e4m3 causal forward B1 H32 N8192 d128", 1, 32, 8192, 128,
                           torch.float8_e4m3fn, 8, causal=True)
FP8_AMP = 16.0
ALL = [TINY_FP32, FWD_N2048, LONG_CAUSAL, TRAIN_N4096, DECODE_L32K, GQA_TRAIN_N4096,
       WINDOW_N8192, GQA_DECODE_L32K, FP8_LONG_CAUSAL]


def _draw(g, shape_per_batch, B, dtype, device):
    out = torch.empty((B,) + tuple(shape_per_batch), dtype=dtype, device=device)
    for b in range(B):
        out[b] = torch.randn(shape_per_batch, generator=g, device=device,
                             dtype=torch.float32).to(dtype)
    return out


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def attention_inputs(B, H, N, d, dtype, seed, device, with_do=False, uniform_head=None):
    """q, k, v (and dO) of shape [B, H, N, d]."""
    g = generator(seed, device)
    q = _draw(g, (H, N, d), B, dtype, device)
    k = _draw(g, (H, N, d), B, dtype, device)
    v = _draw(g, (H, N, d), B, dtype, device)
    if uniform_head is not None:
        k[:, uniform_head] = k[:, uniform_head, :1].expand(-1, N, -1).clone()
    if with_do:
        do = _draw(g, (H, N, d), B, dtype, device)
        return q, k, v, do
    return q, k, v


def gqa_inputs(B, Hq, Hkv, N, d, dtype, seed, device, with_do=False):
    """q [B, Hq, N, d], k, v [B, Hkv, N, d] (and dO [B, Hq, N, d])."""
    g = generator(seed, device)
    q = _draw(g, (Hq, N, d), B, dtype, device)
    k = _draw(g, (Hkv, N, d), B, dtype, device)
    v = _draw(g, (Hkv, N, d), B, dtype, device)
    if with_do:
        return q, k, v, _draw(g, (Hq, N, d), B, dtype, device)
    return q, k, v


def alibi_slopes(H, device):
    """The usual ALiBi slope schedule m_h = 2^(-8 (h + 1) / H), fp32 [H]."""
    h = torch.arange(1, H + 1, dtype=torch.float64)
    return torch.pow(2.0, -8.0 * h / H).to(torch.float32).to(device)


def fp8_inputs(B, Hq, Hkv, N, d, seed, device, amp=FP8_AMP):
    """E4M3 codes as uint8: q [B, Hq, N, d], k, v [B, Hkv, N, d], each drawn
    as fp32 N(0,1) times `amp` and rounded to E4M3 (values stay far below
    the format's 448 limit)."""
    g = generator(seed, device)
    out = []
    for h in (Hq, Hkv, Hkv):
        t = torch.empty((B, h, N, d), dtype=torch.uint8, device=device)
        for b in range(B):
            x = torch.randn((h, N, d), generator=g, device=device, dtype=torch.float32) * amp
            t[b] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        out.append(t)
    return tuple(out)


def decode_gqa_inputs(B, Hq, Hkv, L, d, dtype, seed, device):
    """q [B, Hq, d] and contiguous caches [B, Hkv, L, d]."""
    g = generator(seed, device)
    q = _draw(g, (Hq, d), B, dtype, device)
    kc = _draw(g, (Hkv, L, d), B, dtype, device)
    vc = _draw(g, (Hkv, L, d), B, dtype, device)
    return q, kc, vc


def decode_inputs(B, H, L, d, dtype, seed, device):
    """q [B, H, d] and contiguous caches [B, H, L, d]."""
    g = generator(seed, device)
    q = _draw(g, (H, d), B, dtype, device)
    kc = _draw(g, (H, L, d), B, dtype, device)
    vc = _draw(g, (H, L, d), B, dtype, device)
    return q, kc, vc


def workload_inputs(w: Workload, device):
    if w.dtype == torch.float8_e4m3fn:
        return fp8_inputs(w.B, w.H, w.kv_heads, w.N, w.d, w.seed, device)
    if w.Hkv is not None:
        if w.kind == "decode":
            return decode_gqa_inputs(w.B, w.H, w.Hkv, w.N, w.d, w.dtype, w.seed, device)
        return gqa_inputs(w.B, w.H, w.Hkv, w.N, w.d, w.dtype, w.seed, device,
                          with_do=(w.kind == "train"))
    if w.kind == "decode":
        return decode_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, device)
    return attention_inputs(w.B, w.H, w.N, w.d, w.dtype, w.seed, device,
                            with_do=(w.kind == "train"), uniform_head=w.uniform_head)
