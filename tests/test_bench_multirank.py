"""bench.py's multi-rank path on CPU: two gloo ranks (spawned processes,
rendezvous on 127.0.0.1). Replicas only: the one exchange is the MAX
all-reduce of the timed region, and the reference arm runs on rank 0 alone."""
import argparse
import contextlib
import io
import json
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _worker(rank: int, port: int, q) -> None:
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    try:
        import torch
        import bench
        import workloads
        dist, r, world, _ = bench._dist()
        slowest = bench._max_over_ranks(dist, [3.0, 5.0][r], torch.device("cpu"))
        cfg = workloads.BLOCK_CONFIGS["tiny_stablelm2"]
        args = argparse.Namespace(steps=2, warmup=3)
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            bench.run_reference(args, cfg, r, world, budget_s=5.0)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, r, world, "ok", slowest, out.getvalue()))
    except Exception as e:  # report, do not hang the parent
        q.put((rank, None, None, repr(e), None, ""))


def test_two_gloo_ranks_max_over_ranks_and_rank0_reference():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rk, port, q)) for rk in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, world, status, slowest, _ in got:
        assert status == "ok", status
        assert (r, world) == (rank, 2)
        assert slowest == 5.0            # every rank sees the slowest rank's time
    line = json.loads(got[0][5].strip())
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert got[1][5] == ""               # rank 1 does no work and prints nothing


def test_job_throughput_counts_every_rank():
    import bench
    # 2 ranks x 8192 tokens x 10 steps over the slowest rank's 7 ms
    assert bench._job_throughput(2, 8192, 10, 7.0) == pytest.approx(2 * 8192 * 10 / 0.007)
    assert bench._job_throughput(1, 8192, 10, 7.0) == pytest.approx(8192 * 10 / 0.007)
