"""The multi-rank host logic of bench.py on CPU: two gloo ranks on
127.0.0.1 (world size 2).  The path shards without a data-path collective
(each rank runs its own replica), so what N > 1 adds is the barrier around
the timed loop, the max over ranks of the elapsed time, the whole-job value
and the reference arm running on rank 0 only."""
import json
import os
import socket
import sys
import types

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench as b

    d = b.Dist(world)
    assert (d.world, d.rank, d.local) == (world, rank, rank)
    d.init("gloo")
    d.barrier()
    # each rank's elapsed time differs; every rank must see the slowest
    slowest = d.max(10.0 * (rank + 1), "cpu")
    d.barrier()
    ref = b.run_reference(types.SimpleNamespace(steps=1, warmup=0), d) if rank != 0 else "skip"
    d.close()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "ref_is_none": ref is None}, f)


def test_two_gloo_ranks_barrier_max_and_reference_on_rank0_only(tmp_path):
    world, port = 2, _free_port()
    mp.spawn(_rank, args=(world, port, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(r["slowest"] == 20.0 for r in res)
    # the reference arm does its work (and prints) on rank 0 alone
    assert res[1]["ref_is_none"]


def test_weak_scaling_value():
    # 1e12 FLOP per rank step at 1 ms: 1000 TFLOP/s per rank, N times that for N ranks
    assert bench.weak_scaling_value(1e12, 1, 1.0) == pytest.approx(1000.0)
    assert bench.weak_scaling_value(1e12, 4, 1.0) == pytest.approx(4000.0)
    # the slowest rank sets the step time
    assert bench.weak_scaling_value(1e12, 2, 2.0) == pytest.approx(1000.0)


def test_single_rank_needs_no_process_group():
    d = bench.Dist(1)
    d.init("gloo")          # world 1: no process group is created
    assert d.pg is None
    d.barrier()
    assert d.max(3.5, "cpu") == 3.5
    d.close()
