"""The data-parallel classes with two ranks on one GPU, through the kernels.

Two processes share the GPU, and gloo carries the exchanges on the host, so
no kernel waits on the other rank.  Per rank the test checks:
- WeightCheck: the gathered table against the oracle's fingerprints of both
  ranks' copies, and the same verdict on both ranks (the corrupted copy's rank
  and copy index);
- GradCheck: every rank's gathered statistics against the oracle, the NaN
  rank named on both, then, after the test's own all-reduce (what the training
  framework would do), the reduced gradient's statistics against the oracle on
  the bytes it produced, and the alarm on both ranks.

[AWS] "Check 3: Weight fingerprints, after the optimizer step"; "Check 1:
NaN/Inf gradients, before and after the all-reduce".
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu
LAYOUT = [(64, 32), (32,), (128, 64), (10,), (3, 1000)]
FLIP = (2, 777, 22)  # tensor, element, bit: on rank 1's first copy only


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _copy(seed: int, flip=None):
    """One float32 copy of LAYOUT as host arrays (the same seed on every rank)."""
    rng = np.random.default_rng(seed)
    ts = [(rng.standard_normal(int(np.prod(s))) * 0.02).astype(np.float32).reshape(s) for s in LAYOUT]
    if flip is not None:
        k, e, b = flip
        ts[k].reshape(-1).view(np.uint32)[e] ^= np.uint32(1 << b)
    return ts


def _grads(rank: int):
    rng = np.random.default_rng(50 + rank)
    g = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for n in (5000, 70001)]
    if rank == 1:
        g[1][123] = np.nan
    return g


def _worker(rank, port, copies, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import oracle
    from silent_corruption_checksums_gb300 import dp
    out = {"rank": rank}
    mine = [[torch.from_numpy(a.copy()).cuda() for a in _copy(7, FLIP if (rank == 1 and c == 0) else None)]
            for c in range(copies)]
    wc = dp.WeightCheck(mine)
    res = wc()
    out["verdict"] = res
    every = [_copy(7, FLIP if (r == 1 and c == 0) else None) for r in range(2) for c in range(copies)]
    ref = np.array([[oracle.fingerprint(a.view(np.uint32)) for a in cp] for cp in every], dtype=np.uint64)
    out["table_ok"] = bool(np.array_equal(wc.table.cpu().numpy().view(np.uint64), ref))
    wc.close()

    grads = [torch.from_numpy(a).cuda() for a in _grads(rank)]
    gc = dp.GradCheck(grads)
    before = gc.before_allreduce()
    out["nonfinite"] = before["nonfinite"]
    out["pre_ok"] = []
    for r in range(2):
        ref_r = oracle.grad_stats_multi([a.view(np.uint32) for a in _grads(r)], ["f32", "f32"])
        got = before["stats"][r]
        out["pre_ok"].append(all(got[k] == ref_r[k] for k in ("n_nan", "n_inf", "n_big", "n_elems"))
                             and abs(got["sumsq_finite"] - ref_r["sumsq_finite"]) <= 1e-10 * ref_r["sumsq_finite"])
    for g in grads:  # the framework's all-reduce (average), in place
        dist.all_reduce(g, op=dist.ReduceOp.SUM)
        g.div_(2.0)
    after = gc.after_allreduce()
    reduced = [g.cpu().numpy() for g in grads]
    ref_post = oracle.grad_stats_multi([a.view(np.uint32) for a in reduced], ["f32", "f32"])
    got = after["stats"]
    out["post_ok"] = (all(got[k] == ref_post[k] for k in ("n_nan", "n_inf", "n_big", "n_elems"))
                      and abs(got["sumsq_finite"] - ref_post["sumsq_finite"]) <= 1e-10 * ref_post["sumsq_finite"])
    out["bad"] = after["bad"]
    gc.close()
    q.put(out)
    dist.destroy_process_group()


@pytest.mark.parametrize("copies", [1, 2])
def test_two_ranks_on_one_gpu(copies):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, copies, q)) for r in range(2)]
    for p in procs:
        p.start()
    outs = sorted((q.get(timeout=300) for _ in procs), key=lambda o: o["rank"])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for o in outs:
        assert o["table_ok"]
        if copies == 1:  # two copies that disagree: detected, no rank named
            assert o["verdict"] == {"diverged": True, "suspects": None, "suspect_replicas": None}
        else:  # four copies: rank 1's first copy (gathered copy 2) is named, and so is rank 1
            assert o["verdict"] == {"diverged": True, "suspects": [1], "suspect_replicas": [2]}
        assert o["nonfinite"] == [1]
        assert o["pre_ok"] == [True, True]
        assert o["post_ok"] and o["bad"] is True
