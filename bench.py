#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300 (one JSON line).

One step = one pass of the whole training hot path on the workload
"bf16 causal forward+backward B8 H32 N4096 d128": the fused forward kernel
(Q block on chip, K/V tiles streamed, online softmax, O and LSE written once)
followed by the recomputation backward (D = rowsum(dO*O), the dK/dV/dQ kernel,
the dQ conversion).  ``value`` is the attention TFLOP/s of that step, counted
as 4 B H N^2 d for the forward (halved under the causal mask) plus 2.5 times
that for the backward, summed over every rank.

The same line carries:
  roofline      the dominant kernel (backward dK/dV/dQ) against the measured
                burst bf16 tensor peak (the timed loop is short and runs at
                the full SM clock), timed with events recorded by the library
                immediately around that kernel;
  e2e           the same metric through the public API with the step's inputs
                copied from pinned host memory and dQ, dK, dV copied back;
  targets       the forward kernel alone on "bf16 causal forward B1 H32 N8192"
                and on "bf16 forward B4 H16 N2048" (causal and not), against
                the burst bf16 peak, and split-KV decode on "B64 H32 Lkv32768"
                in KV GB/s against the measured HBM copy bandwidth; then the
                grouped-query forward and backward kernels (B8 Hq32 Hkv8
                N4096 causal), the causal sliding-window forward (w = 1024,
                B1 H32 N8192), grouped-query decode (B64 Hq32 Hkv8
                Lkv32768) and the fp8 (E4M3) causal forward B1 H32 N8192
                against the fp8 dense peak;
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload;
  clocks        SM clocks and throttle reasons sampled during the timed loop.

``--impl reference`` times the oracle instead (the only reference this method
has), on host cores, for the same metric and workload.

Under torchrun each rank runs its own replica of the workload (weak scaling;
the (batch, head) units are independent, so no collective touches the data).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s and % of GB300 BF16 peak; decode KV HBM GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- distributed
class Dist:
    def __init__(self, want_gpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.want = want_gpus
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device) -> float:
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def weak_scaling_value(flops_per_rank_step: float, world: int, ms_step_max: float) -> float:
    """Whole-job TFLOP/s: every rank runs the same replica, so the work of all
    ranks in one step over the slowest rank's step time."""
    return flops_per_rank_step * world / (ms_step_max * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- helpers
def lib_event():
    """A timing event the library can record: torch creates events lazily,
    so record it once here to make its handle exist."""
    import torch

    e = torch.cuda.Event(enable_timing=True)
    e.record()
    return e


def kernel_source_hash(name: str, upto: str | None = None) -> str:
    """Hash of a kernel's source: its file up to the marker `upto` (the
    kernels of a file come before their launchers, so a change to a later
    kernel or to host code leaves the hash alone) plus the shared device
    header."""
    csrc = os.path.join(ROOT, "exact_attention_84_gb300", "csrc")
    with open(os.path.join(csrc, name), "rb") as f:
        text = f.read()
    if upto is not None:
        cut = text.find(upto.encode())
        if cut < 0:
            return "marker-missing"
        text = text[:cut]
    with open(os.path.join(csrc, "fa_device.cuh"), "rb") as f:
        text += f.read()
    return hashlib.sha256(text).hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel
    source is unchanged since the capture; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(key)
    if not rec or rec.get("source_sha256_16") != kernel_source_hash(rec["file"],
                                                                     rec.get("hash_upto")):
        return None
    return rec.get("dram_bytes_per_launch")


def cpu_oracle_sample(q, k, v, do, heads, scale, causal, budget_s=10.0):
    """Time the fp64 oracle (forward + backward) on (b, h) pairs taken in the
    order of `heads` until `budget_s` seconds of wall time have been spent
    (at least one pair).  Returns (pairs done, wall s, process CPU s)."""
    import numpy as np

    import oracle.attention as orc

    wall = cpu = 0.0
    done = 0
    for b, h in heads:
        qh, kh, vh, doh = (t[b, h].float().cpu().numpy().astype(np.float64)[None]
                           for t in (q, k, v, do))
        c0 = time.process_time()
        t0 = time.perf_counter()
        orc.attention_forward(qh, kh, vh, scale, causal)
        orc.attention_backward(qh, kh, vh, doh, scale, causal)
        wall += time.perf_counter() - t0
        cpu += time.process_time() - c0
        done += 1
        if wall >= budget_s:
            break
    return done, wall, cpu


# ---------------------------------------------------------------- our arm
def run_ours(args, dist: Dist):
    import numpy as np
    import torch

    from exact_attention_84_gb300 import _lib, accounting as acc, api, inputs

    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    w = inputs.TRAIN_N4096
    B, H, N, d = w.B, w.H, w.N, w.d
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = inputs.attention_inputs(B, H, N, d, w.dtype, w.seed + 1000 * dist.rank, dev,
                                          with_do=True)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = _lib.fa_workspace_size(_lib.FA_OP_BACKWARD, B, H, N, d, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fwd_fl = acc.forward_flops(B, H, N, d, True)
    bwd_fl = acc.backward_flops(B, H, N, d, True)

    def step(ev=None):
        if ev is not None:
            _lib.check(_lib.fa_set_timing_events(ev[0].cuda_event, ev[1].cuda_event))
        _lib.check(_lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, scale, 1, sh))
        if ev is not None:
            _lib.check(_lib.fa_set_timing_events(ev[2].cuda_event, ev[3].cuda_event))
        _lib.check(_lib.fa_backward_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale, 1,
                                       ws.data_ptr(), ws_bytes, sh))
        if ev is not None:
            _lib.check(_lib.fa_set_timing_events(None, None))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if api.device_status() != 0:
        raise RuntimeError("kernel timeout during warm-up: " + _lib.fa_last_error())

    evs = [[lib_event() for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dist.local)
    dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = dist.max(total_ms, dev)
    ms_step = total_ms / args.steps
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    value = weak_scaling_value(fwd_fl + bwd_fl, dist.world, ms_step)

    # --- end to end through the public API with host buffers.  Every step
    # copies its four inputs in from pinned host memory and its three
    # gradients back out; as in a training loop, step i+1's upload and step
    # i-1's download run on their own streams while step i computes
    # (double-buffered device tensors, ordered by events).
    pin_in = [t.cpu().pin_memory() for t in (q, k, v, do)]
    pin_out = [[torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3)]
               for _ in range(2)]
    dev_in = [[torch.empty_like(t) for t in (q, k, v, do)] for _ in range(2)]
    dev_o = [(torch.empty_like(q), torch.empty_like(lse)) for _ in range(2)]
    dev_g = [[torch.empty_like(q) for _ in range(3)] for _ in range(2)]
    s_h2d, s_comp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def fresh_event():
        e = torch.cuda.Event()
        e.record()
        return e

    ev_in = [fresh_event() for _ in range(2)]
    ev_used = [fresh_event() for _ in range(2)]
    ev_out = [fresh_event() for _ in range(2)]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_h2d):
            s_h2d.wait_event(ev_used[b])        # step i-2 finished with these buffers
            for d_, h_ in zip(dev_in[b], pin_in):
                d_.copy_(h_, non_blocking=True)
            ev_in[b].record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[b])
            s_comp.wait_event(ev_out[b])         # step i-2's gradients are on the host
            qd, kd, vd, dod = dev_in[b]
            od, lsed = api.forward(qd, kd, vd, causal=True, scale=scale, out=dev_o[b][0],
                                   lse=dev_o[b][1])
            api.backward(qd, kd, vd, od, lsed, dod, causal=True, scale=scale, workspace=ws,
                         out=dev_g[b])
            ev_used[b].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(ev_used[b])
            for h_, d_ in zip(pin_out[b], dev_g[b]):
                h_.copy_(d_, non_blocking=True)
            ev_out[b].record(s_d2h)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    dist.barrier()
    e0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = dist.max(time.perf_counter() - e0, dev) / args.steps
    h2d = sum(t.numel() * t.element_size() for t in pin_in)
    d2h = sum(t.numel() * t.element_size() for t in pin_out[0])
    e2e = {"value": round((fwd_fl + bwd_fl) * dist.world / e2e_s / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_s * 1e3, 3),
           "overlap": "inputs in, compute, gradients out on three streams, double-buffered"}
    # the last step's gradients came back through the host buffers: spot-check
    if not torch.equal(pin_out[(args.steps - 1) % 2][0], dev_g[(args.steps - 1) % 2][0].cpu()):
        raise RuntimeError("end-to-end gradients did not reach the host")
    del pin_in, pin_out, dev_in, dev_o, dev_g

    # --- roofline of the dominant kernel (the backward dK/dV/dQ kernel)
    # The timed loop is well under a second at the full SM clock, so the
    # denominator is the burst peak (a GEMM timed alone); the sustained peak,
    # taken over seconds under the power cap at a lower clock, is kept as a
    # labelled secondary figure.
    peak_burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    ach = bwd_fl / (bwd_ms * 1e-3) / 1e12
    roofline = {"kernel": "bwd_main_kernel (dK, dV, dQ)", "bound": "tensor",
                "achieved": round(ach, 1), "peak": peak_burst, "unit": "TFLOP/s",
                "frac": round(ach / peak_burst, 4),
                "peak_kind": f"bf16 dense, burst ({peak_src})",
                "frac_of_sustained": round(ach / peak_sus, 4), "sustained_peak": peak_sus,
                "flops_per_launch": bwd_fl, "ms_per_launch": round(bwd_ms, 4),
                "traffic": recorded_traffic("bwd_main_kernel")}
    fwd_ach = fwd_fl / (fwd_ms * 1e-3) / 1e12
    step_parts = {"forward_ms": round(fwd_ms, 4), "forward_tflops": round(fwd_ach, 1),
                  "backward_main_ms": round(bwd_ms, 4),
                  "backward_call_other_ms": round(ms_step - fwd_ms - bwd_ms, 4)}

    targets = None
    if not args.no_targets:
        targets = measure_targets(args, dev, peaks, peak_src)

    cpu = None
    if dist.rank == 0 and not args.no_cpu:
        order = [(b, h) for b in range(B) for h in range(H)]
        order = [order[i] for i in np.random.default_rng(3).permutation(len(order))]
        n_done, wall, cput = cpu_oracle_sample(q, k, v, do, order, scale, True,
                                               budget_s=args.cpu_seconds)
        per_head = acc.forward_flops(1, 1, N, d, True) + acc.backward_flops(1, 1, N, d, True)
        cpu = {"value": round(per_head * n_done / wall / 1e12, 6), "unit": "TFLOP/s",
               "cores": os.cpu_count(), "threads_busy": round(cput / wall, 1), "kind": "oracle",
               "sample": f"fp64 forward+backward of {n_done} of the {B * H} heads "
                         f"(N={N}, causal; seeded random heads, about {args.cpu_seconds:g} s "
                         f"of work), {wall:.1f} s wall"}

    dist.barrier()
    dist.close()
    if dist.rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16)",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "causal": True,
                   "global_batch": B * dist.world, "seq_len": N,
                   "parallelism": f"independent replicas x{dist.world} (no collective)",
                   "l2": "inputs larger than L2 (268 MB per tensor), no flush"},
        "gpu_launches": 4 * args.steps,
        "step": step_parts, "roofline": roofline, "e2e": e2e, "targets": targets,
        "cpu_baseline": cpu, "clocks": clk,
        # O(N) memory: the only device memory beyond inputs and outputs is the
        # backward workspace (fp32 dQ accumulator + two padded stat rows), no
        # N x N buffer; per head against the N^2 bf16 score matrix it avoids
        "memory": {"forward_workspace_bytes": 0, "backward_workspace_bytes": ws_bytes,
                   "backward_workspace_bytes_per_head": ws_bytes // (B * H),
                   "n2_bf16_bytes_per_head": N * N * 2},
    }


def measure_targets(args, dev, peaks, peak_src):
    """Each kernel alone on its own workload, events recorded by the library
    around the kernel; L2 flushed between iterations where inputs fit in L2."""
    import torch

    from exact_attention_84_gb300 import _lib, accounting as acc, inputs

    sh = torch.cuda.current_stream().cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    iters = max(5, args.target_iters)

    def time_kernel(call, do_flush):
        ts = []
        for i in range(3 + iters):
            if do_flush:
                flush.zero_()
            a, b = lib_event(), lib_event()
            _lib.check(_lib.fa_set_timing_events(a.cuda_event, b.cuda_event))
            call()
            _lib.check(_lib.fa_set_timing_events(None, None))
            torch.cuda.synchronize()
            if i >= 3:
                ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    out = {}
    for w, causal, key in ((inputs.LONG_CAUSAL, True, "forward_causal_B1_H32_N8192"),
                           (inputs.FWD_N2048, True, "forward_causal_B4_H16_N2048"),
                           (inputs.FWD_N2048, False, "forward_B4_H16_N2048")):
        q, k, v = inputs.workload_inputs(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
        fits_l2 = 4 * q.numel() * q.element_size() < 129e6 * 1.5
        ms = time_kernel(lambda: _lib.check(_lib.fa_forward(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H,
            w.N, w.d, 1 / math.sqrt(w.d), int(causal), sh)), fits_l2)
        fl = acc.forward_flops(w.B, w.H, w.N, w.d, causal)
        t = fl / (ms * 1e-3) / 1e12
        out[key] = {"ms": round(ms, 4), "tflops": round(t, 1), "frac": round(t / burst, 4),
                    "peak": burst, "peak_kind": f"bf16 dense, burst ({peak_src})",
                    "l2_flush": bool(fits_l2)}
        del q, k, v, o, lse
    w = inputs.DECODE_L32K
    q, kc, vc = inputs.workload_inputs(w, dev)
    o = torch.empty_like(q)
    best = None
    for s in args.decode_splits:
        ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_DECODE, w.B, w.H, w.N, w.d, s),
                         dtype=torch.uint8, device=dev)
        ms = time_kernel(lambda: _lib.check(_lib.fa_decode_ex(
            q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, w.B, w.H, w.N, w.d,
            s, 1 / math.sqrt(w.d), ws.data_ptr(), ws.numel(), sh)), False)
        gbs = acc.decode_kv_bytes(w.B, w.H, w.N, w.d) / (ms * 1e-3) / 1e9
        rec = {"num_splits": s, "ms": round(ms, 4), "kv_gbs": round(gbs, 1),
               "frac": round(gbs / hbm, 4)}
        if best is None or gbs > best["kv_gbs"]:
            best = rec
    out["decode_B64_H32_L32768"] = dict(best, peak=hbm, unit="GB/s",
                                        peak_kind=f"HBM copy ({peak_src})",
                                        timed="whole call: split kernel + combine kernel",
                                        bytes_per_launch=acc.decode_kv_bytes(w.B, w.H, w.N, w.d))
    del q, kc, vc, o

    # grouped query heads (4 per key/value head): forward and backward kernels
    w = inputs.GQA_TRAIN_N4096
    q, k, v, do = inputs.workload_inputs(w, dev)
    hkv, scale = w.kv_heads, 1 / math.sqrt(w.d)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_BACKWARD, w.B, w.H, w.N, w.d, 0),
                     dtype=torch.uint8, device=dev)
    fwd = lambda: _lib.check(_lib.fa_forward_gqa(  # noqa: E731
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, hkv,
        w.N, w.d, scale, 1, 0, None, sh))
    bwd = lambda: _lib.check(_lib.fa_backward_gqa(  # noqa: E731
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, hkv, w.N, w.d, scale, 1, 0,
        None, 0, ws.data_ptr(), ws.numel(), sh))
    fl = acc.forward_flops(w.B, w.H, w.N, w.d, True)
    for key, call, flops in (("forward_gqa_causal_B8_Hq32_Hkv8_N4096", fwd, fl),
                             ("backward_gqa_causal_B8_Hq32_Hkv8_N4096", bwd, 2.5 * fl)):
        ms = time_kernel(call, False)
        t = flops / (ms * 1e-3) / 1e12
        out[key] = {"ms": round(ms, 4), "tflops": round(t, 1), "frac": round(t / burst, 4),
                    "peak": burst, "peak_kind": f"bf16 dense, burst ({peak_src})",
                    "l2_flush": False}
    del q, k, v, do, o, lse, dq, dk, dv, ws

    # causal sliding window: FLOPs of the visible (query, key) pairs only
    w = inputs.WINDOW_N8192
    q, k, v = inputs.workload_inputs(w, dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    ms = time_kernel(lambda: _lib.check(_lib.fa_forward_gqa(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.H,
        w.N, w.d, 1 / math.sqrt(w.d), 1, w.window, None, sh)), False)
    fl = acc.masked_forward_flops(w.B, w.H, w.N, w.d, True, w.window)
    t = fl / (ms * 1e-3) / 1e12
    out["forward_window1024_B1_H32_N8192"] = {
        "ms": round(ms, 4), "tflops": round(t, 1), "frac": round(t / burst, 4), "peak": burst,
        "peak_kind": f"bf16 dense, burst ({peak_src})", "l2_flush": False,
        "flops": "4 d per visible (query, key) pair"}
    del q, k, v, o, lse

    # FP8 (E4M3) causal forward: the main kernel against the fp8 dense peak
    # (the measured bf16 peak times the nominal fp8/bf16 ratio 4.5/2.25), and
    # the whole call (V transposition included)
    w = inputs.FP8_LONG_CAUSAL
    q8, k8, v8 = inputs.workload_inputs(w, dev)
    o = torch.empty(q8.shape, device=dev, dtype=torch.bfloat16)
    lse = torch.empty(q8.shape[:3], device=dev, dtype=torch.float32)
    ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_FORWARD_FP8, w.B, w.H, w.N, w.d, 0),
                     dtype=torch.uint8, device=dev)
    ds = 1.0 / inputs.FP8_AMP
    call = lambda: _lib.check(_lib.fa_forward_fp8(  # noqa: E731
        q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H,
        w.H, w.N, w.d, 1 / math.sqrt(w.d), ds, ds, ds, 1, 0, None, ws.data_ptr(), ws.numel(),
        sh))
    ms = time_kernel(call, False)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    a, b = lib_event(), lib_event()
    a.record()
    for _ in range(iters):
        call()
    b.record()
    torch.cuda.synchronize()
    ms_call = a.elapsed_time(b) / iters
    fl = acc.forward_flops(w.B, w.H, w.N, w.d, True)
    fp8_peak = 2.0 * burst
    t = fl / (ms * 1e-3) / 1e12
    out["forward_fp8_causal_B1_H32_N8192"] = {
        "ms": round(ms, 4), "tflops": round(t, 1), "frac": round(t / fp8_peak, 4),
        "peak": fp8_peak, "peak_kind": f"fp8 dense = 2 x bf16 burst ({peak_src}), nominal ratio",
        "call_ms": round(ms_call, 4),
        "call_tflops": round(fl / (ms_call * 1e-3) / 1e12, 1), "l2_flush": False}
    del q8, k8, v8, o, lse, ws

    # grouped-query decode: the cache (Hkv heads) read once for all query heads
    w = inputs.GQA_DECODE_L32K
    q, kc, vc = inputs.workload_inputs(w, dev)
    o = torch.empty_like(q)
    hkv = w.kv_heads
    kv_bytes = acc.decode_kv_bytes(w.B, hkv, w.N, w.d)
    best = None
    for s in args.decode_splits:
        ws = torch.empty(_lib.fa_workspace_size(_lib.FA_OP_DECODE, w.B, w.H, w.N, w.d, s),
                         dtype=torch.uint8, device=dev)
        ms = time_kernel(lambda: _lib.check(_lib.fa_decode_gqa(
            q.data_ptr(), kc.data_ptr(), vc.data_ptr(), o.data_ptr(), None, w.B, w.H, hkv, w.N,
            w.d, s, 1 / math.sqrt(w.d), None, ws.data_ptr(), ws.numel(), sh)), False)
        gbs = kv_bytes / (ms * 1e-3) / 1e9
        rec = {"num_splits": s, "ms": round(ms, 4), "kv_gbs": round(gbs, 1),
               "frac": round(gbs / hbm, 4)}
        if best is None or gbs > best["kv_gbs"]:
            best = rec
    out["decode_gqa_B64_Hq32_Hkv8_L32768"] = dict(best, peak=hbm, unit="GB/s",
                                                  peak_kind=f"HBM copy ({peak_src})",
                                                  timed="whole call: split kernel + combine kernel",
                                                  bytes_per_launch=kv_bytes)
    return out


# ---------------------------------------------------------------- reference arm
def run_reference(args, dist: Dist):
    """The oracle (plain fp64 CPU definition) on the host cores, same metric
    and workload, each step a bounded sample: one (b, h) head of the training
    workload, forward + backward."""
    import numpy as np

    from exact_attention_84_gb300 import accounting as acc
    from exact_attention_84_gb300 import inputs
    import oracle.attention as orc
    import torch

    if dist.rank != 0:
        return None
    w = inputs.TRAIN_N4096
    N, d = w.N, w.d
    scale = 1 / math.sqrt(d)
    q, k, v, do = inputs.attention_inputs(1, 1, N, d, w.dtype, w.seed, "cpu", with_do=True)
    qh, kh, vh, doh = (t.float().numpy().astype(np.float64) for t in (q, k, v, do))

    def step():
        orc.attention_forward(qh, kh, vh, scale, True)
        orc.attention_backward(qh, kh, vh, doh, scale, True)

    for _ in range(args.warmup):
        step()
    c0 = time.process_time()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    wall = time.perf_counter() - t0
    cput = time.process_time() - c0
    fl = acc.forward_flops(1, 1, N, d, True) + acc.backward_flops(1, 1, N, d, True)
    value = fl * args.steps / wall / 1e12
    sample = f"fp64 oracle forward+backward of one (b,h) head of {w.name} per step"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-rounded, computed in fp64)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": N, "d": d, "causal": True,
                   "sample": "1 head per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "threads_busy": round(cput / wall, 1), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-targets", action="store_true", help="skip the per-kernel targets")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-time budget of the CPU oracle sample")
    ap.add_argument("--target-iters", type=int, default=10)
    ap.add_argument("--decode-splits", type=int, nargs="+", default=[1, 2, 4, 8])
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    dist = Dist(args.gpus)
    if args.impl == "reference":
        res = run_reference(args, dist)
    else:
        res = run_ours(args, dist)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
