"""The N > 1 path of bench.py on the CPU: two gloo ranks (world size 2).

Each GPU runs an independent replica (every (batch row, head) is independent,
so the work shards with no collective on the data path); the only
cross-rank steps are the rendezvous, the barriers around the timed region,
the max of the ranks' times and the whole-job throughput.  Two spawned
processes run exactly those functions of bench.py over gloo on
127.0.0.1 and check that both ranks see the slowest rank's time, that the
whole-job value counts both ranks' units, and that the reference arm does
its work on rank 0 only (rank 1 returns at once and prints nothing).
"""
import argparse
import contextlib
import io
import json
import os
import socket
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, local = bench.dist_setup(backend="gloo")  # the same backend on every machine
    bench.barrier(w)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_ms, w, torch.device("cpu"))
    rate = bench.whole_job_rate(1000.0, w, slowest / 1e3)
    printed = ""
    if rank != 0:
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(argparse.Namespace(steps=1, warmup=3))
        printed = buf.getvalue()
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "slowest": slowest, "rate": rate, "printed": printed}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r
        assert d["slowest"] == 15.0                    # max over ranks, seen by both
        assert abs(d["rate"] - 2000.0 / 0.015) < 1e-6  # both ranks' units / slowest time
    assert res[1]["printed"] == ""                      # reference arm: rank 0 only


def test_whole_job_rate_single_rank():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(8192.0, 1, 0.5) == 16384.0
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
