"""fp64 CPU oracle for exact attention (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs may
import this package; the CUDA library never does.
"""

from .attention import (  # noqa: F401
    attention_backward_gqa,
    attention_decode_gqa,
    attention_forward_gqa,
    attention_backward,
    attention_decode,
    attention_forward,
    attention_forward_rows,
    online_softmax_stats,
    tile_merged_attention_row,
)
from .fp8 import attention_forward_fp8, decode_e4m3  # noqa: F401
