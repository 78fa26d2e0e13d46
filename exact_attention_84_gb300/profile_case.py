"""Run one kernel family on a profiling-sized workload, for ncu captures.

    python -m exact_attention_84_gb300.profile_case CASE [--launches K]

Workloads (inputs larger than the 129 MB L2, a few GB on the device at most):
  fwd     bf16 causal forward B1 H32 N8192 d128 (the long-context workload itself)
  fwd_nc  bf16 non-causal forward B4 H16 N2048 d128
  bwd     bf16 causal backward B2 H32 N4096 d128 (a quarter of the training
          workload's heads; its traffic scales with the heads)
  decode  bf16 split-KV decode B4 H32 Lkv32768 d128, 8 splits (1/16 of the
          decode workload's sequences)
  fwd_win bf16 causal sliding-window (w=1024) forward B1 H32 N8192 d128 (the
          windowed workload itself)
  bwd_gqa bf16 causal GQA backward B2 Hq32 Hkv8 N4096 d128 (a quarter of the
          GQA training workload)
  dec_gqa bf16 GQA split-KV decode B4 Hq32 Hkv8 Lkv32768 d128, 8 splits (1/16
          of the GQA decode workload's sequences)
  fwd_fp8 fp8 (E4M3) causal forward B1 H32 N8192 d128 (the fp8 workload
          itself; the call runs the V transposition, then the forward)
  fwd_fp32 fp32 forward B1 H1 N256 d64 (the tiny fp32 workload itself)
  bwd_det bf16 causal deterministic backward B2 H32 N4096 d128 (dK/dV
          kernel without dQ, then the query-stationary dQ kernel)
One warm-up launch precedes the K profiled ones.  Prints the mean device
time per launch measured with CUDA events (not a bench value under ncu).
"""

from __future__ import annotations

import argparse
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    from exact_attention_84_gb300 import _lib, inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["fwd", "fwd_nc", "bwd", "decode", "fwd_win", "bwd_gqa",
                                     "dec_gqa", "fwd_fp8", "fwd_fp32", "bwd_det"])
    ap.add_argument("--launches", type=int, default=2)
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    sh = torch.cuda.current_stream().cuda_stream
    d = 128
    scale = 1 / math.sqrt(d)
    if a.case in ("fwd", "fwd_nc"):
        B, H, N, causal, seed = (1, 32, 8192, 1, 2) if a.case == "fwd" else (4, 16, 2048, 0, 1)
        q, k, v = inputs.attention_inputs(B, H, N, d, torch.bfloat16, seed, dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)

        def call():
            _lib.check(_lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, H, N, d, scale, causal, sh))
    elif a.case == "bwd":
        B, H, N = 2, 32, 4096
        q, k, v, do = inputs.attention_inputs(B, H, N, d, torch.bfloat16, 3, dev, with_do=True)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
        _lib.check(_lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, scale, 1, sh))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nbytes = _lib.fa_workspace_size(_lib.FA_OP_BACKWARD, B, H, N, d, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def call():
            _lib.check(_lib.fa_backward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                           dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale, 1,
                                           ws.data_ptr(), nbytes, sh))
    elif a.case == "bwd_det":
        B, H, N = 2, 32, 4096
        q, k, v, do = inputs.attention_inputs(B, H, N, d, torch.bfloat16, 3, dev, with_do=True)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
        _lib.check(_lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, scale, 1, sh))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nbytes = _lib.fa_workspace_size(_lib.FA_OP_BACKWARD, B, H, N, d, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def call():
            _lib.check(_lib.fa_backward_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, H,
                                            N, d, scale, 1, 0, None, 1, ws.data_ptr(), nbytes,
                                            sh))
    elif a.case == "fwd_fp8":
        B, H, N = 1, 32, 8192
        q8, k8, v8 = inputs.fp8_inputs(B, H, H, N, d, 8, dev)
        o = torch.empty((B, H, N, d), device=dev, dtype=torch.bfloat16)
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
        nbytes = _lib.fa_workspace_size(_lib.FA_OP_FORWARD_FP8, B, H, N, d, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        ds = 1.0 / inputs.FP8_AMP

        def call():
            _lib.check(_lib.fa_forward_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(),
                                           o.data_ptr(), lse.data_ptr(), B, H, H, N, d, scale,
                                           ds, ds, ds, 1, 0, None, ws.data_ptr(), nbytes, sh))
    elif a.case == "fwd_fp32":
        B, H, N, d32 = 1, 1, 256, 64
        q, k, v = inputs.attention_inputs(B, H, N, d32, torch.float32, 0, dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)

        def call():
            _lib.check(_lib.fa_forward_fp32(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse.data_ptr(), B, H, N, d32,
                                            1 / math.sqrt(d32), 0, sh))
    elif a.case == "fwd_win":
        B, H, N, W = 1, 32, 8192, 1024
        q, k, v = inputs.attention_inputs(B, H, N, d, torch.bfloat16, 6, dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)

        def call():
            _lib.check(_lib.fa_forward_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), B, H, H, N, d, scale, 1, W, None,
                                           sh))
    elif a.case == "bwd_gqa":
        B, Hq, Hkv, N = 2, 32, 8, 4096
        q, k, v, do = inputs.gqa_inputs(B, Hq, Hkv, N, d, torch.bfloat16, 5, dev, with_do=True)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), device=dev, dtype=torch.float32)
        _lib.check(_lib.fa_forward_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, Hq, Hkv, N, d, scale, 1, 0, None, sh))
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        nbytes = _lib.fa_workspace_size(_lib.FA_OP_BACKWARD, B, Hq, N, d, 0)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def call():
            _lib.check(_lib.fa_backward_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq,
                                            Hkv, N, d, scale, 1, 0, None, 0, ws.data_ptr(),
                                            nbytes, sh))
    elif a.case == "dec_gqa":
        B, Hq, Hkv, L, S = 4, 32, 8, 32768, 8
        q, kc, vc = inputs.decode_gqa_inputs(B, Hq, Hkv, L, d, torch.bfloat16, 7, dev)
        o = torch.empty_like(q)
        nbytes = _lib.fa_workspace_size(_lib.FA_OP_DECODE, B, Hq, L, d, S)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def call():
            _lib.check(_lib.fa_decode_gqa(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                          None, B, Hq, Hkv, L, d, S, scale, None, ws.data_ptr(),
                                          nbytes, sh))
    else:
        B, H, L, S = 4, 32, 32768, 8
        q, kc, vc = inputs.decode_inputs(B, H, L, d, torch.bfloat16, 4, dev)
        o = torch.empty_like(q)
        nbytes = _lib.fa_workspace_size(_lib.FA_OP_DECODE, B, H, L, d, S)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def call():
            _lib.check(_lib.fa_decode_ex(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(),
                                         None, B, H, L, d, S, scale, ws.data_ptr(), nbytes, sh))
    call()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    e.record()          # torch creates events lazily; make both handles exist
    _lib.check(_lib.fa_set_timing_events(s.cuda_event, e.cuda_event))
    tot = 0.0
    for _ in range(a.launches):
        call()
        torch.cuda.synchronize()
        tot += s.elapsed_time(e)
    _lib.check(_lib.fa_set_timing_events(None, None))
    status = _lib.fa_get_device_status(sh)
    print(f"{a.case}: {tot / a.launches:.4f} ms per launch (main kernel), status {status}")
    sys.exit(0 if status == 0 else 1)


if __name__ == "__main__":
    main()
