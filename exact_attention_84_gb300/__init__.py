"""Exact attention (FlashAttention-style fused forward, recomputation
backward, split-KV decode) for one NVIDIA GB300, behind a C ABI (libfa.so)."""

from . import _lib  # noqa: F401
from .api import backward, decode, device_status, forward  # noqa: F401
