"""The benchmark's multi-rank host logic with two gloo ranks on the CPU:
max-over-ranks timing, whole-job throughput, and rank 0 alone printing the
reference arm's line."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, local = bench.dist_env()
    bench.barrier(w)
    mine = 1.5 if rank == 0 else 4.0  # ms per step seen by this rank
    slowest = bench.max_over_ranks(mine, w)
    rate = bench.whole_job_rate(12_475_438_080, w, slowest)
    q.put((rank, r, w, slowest, rate))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, slowest, rate in out:
        assert r == rank and w == 2
        assert slowest == 4.0
        assert rate == pytest.approx(2 * 12_475_438_080 / 4e-3 / 1e9)


def test_reference_arm_prints_on_rank_zero_only(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(bench_args(steps=1, warmup=0))
    assert capsys.readouterr().out == ""


def bench_args(**kw):
    import argparse
    ns = argparse.Namespace(gpus=2, steps=1, warmup=0, impl="reference", chunk_bytes=0, quick=False, traffic=None,
                            layers=24, only=None)
    for k, v in kw.items():
        setattr(ns, k, v)
    return ns
