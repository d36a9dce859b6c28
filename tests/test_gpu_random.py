"""Randomized parity sweep: many seeded plans with random tensor counts, sizes,
element widths, start offsets, chunk sizes and corruptions, each checked
against the oracle (fingerprint, xorsum, vote, grad stats)."""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import fp_table, host_bits, oracle_fp_table, stats_match

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.uint8, torch.int16, torch.bfloat16, torch.float16, torch.float32, torch.float64]
NAMES = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _random_plan(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 9))
    T = int(rng.integers(1, 40))
    float_only = bool(rng.integers(0, 2))
    pool = DTYPES[2:5] if float_only else DTYPES
    specs = []
    for _ in range(T):
        dt = pool[int(rng.integers(len(pool)))]
        n = int(np.floor(np.exp(rng.uniform(0, np.log(300_000)))))
        if rng.random() < 0.05:
            n = 0
        specs.append((dt, n, int(rng.integers(0, 9))))  # dtype, numel, start offset in elements
    gen = W.generator(seed, DEV)
    base = []
    for dt, n, off in specs:
        es = torch.empty(0, dtype=dt).element_size()
        raw = torch.randint(0, 256, ((n + off) * es,), generator=gen, device=DEV, dtype=torch.int64).to(torch.uint8)
        if dt.is_floating_point:
            buf = W.normal((n + off,), 0.02, dt, gen, DEV)
        else:
            buf = raw.view(dt)
        base.append(buf[off:off + n])
    reps = []
    for r in range(R):
        ts = []
        for t, (dt, n, off) in zip(base, specs):
            buf = torch.empty(n + off, dtype=dt, device=DEV)
            buf[off:].copy_(t)
            ts.append(buf[off:])
        reps.append(ts)
    for _ in range(int(rng.integers(0, 4))):
        r, k = int(rng.integers(R)), int(rng.integers(T))
        if reps[r][k].numel():
            es = reps[r][k].element_size()
            W.xor_element(reps[r][k], int(rng.integers(reps[r][k].numel())), 1 << int(rng.integers(8 * es)))
    chunk = int(2 ** rng.integers(12, 16))
    return reps, chunk, float_only


@pytest.mark.parametrize("seed", range(24))
def test_random_plans(sdc, seed):
    reps, chunk, float_only = _random_plan(1000 + seed)
    plan = sdc.Plan(reps, chunk_bytes=chunk)
    fp = plan.fingerprint()
    ref = oracle_fp_table(reps)
    assert fp_table(fp) == ref
    suspect, mask, summary = sdc.vote(fp)
    rs, rm, rsumm = oracle.vote(ref)
    assert suspect.cpu().tolist() == rs
    assert [int(x) & ((1 << 64) - 1) for x in mask.cpu().numpy().view(np.uint64)] == rm
    assert sdc.pages_verdict(sdc.decode_summary(summary)) == oracle.pages_verdict(rsumm)
    xs = plan.xorsum().cpu().numpy().view(np.uint64)
    for r, ts in enumerate(reps):
        for k, t in enumerate(ts):
            assert int(xs[r, k]) == oracle.xorsum(host_bits(t))
    if float_only:
        stats = sdc.decode_stats(plan.grad_scan())
        for r, ts in enumerate(reps):
            stats_match(stats[r], oracle.grad_stats_multi([host_bits(t) for t in ts], [NAMES[t.dtype] for t in ts]))


def test_weight_check_in_a_cuda_graph(sdc):
    """The whole weight check (scan, combine, vote) captured once and replayed."""
    w = W.tiny(DEV, seed=4)
    plan = sdc.Plan(w["replicas"])
    T = len(w["replicas"][0])
    fp = torch.empty((3, T, 2), dtype=torch.int64, device=DEV)
    out = (torch.empty(T, dtype=torch.int32, device=DEV), torch.empty(T, dtype=torch.int64, device=DEV),
           torch.empty(sdc.VOTE_SUMMARY_DTYPE.itemsize, dtype=torch.uint8, device=DEV))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.fingerprint(out=fp, stream=s)  # warm up outside the capture
        sdc.vote(fp, stream=s, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.fingerprint(out=fp, stream=s)
        sdc.vote(fp, stream=s, out=out)
    fp.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert fp_table(fp) == oracle_fp_table(w["replicas"])
    assert sdc.pages_verdict(sdc.decode_summary(out[2])) == {"diverged": True, "suspects": [1]}
    # corrupt another replica between replays: the same graph sees it
    W.xor_element(w["replicas"][2][0], 3, 1 << 30)
    g.replay()
    torch.cuda.synchronize()
    summ = sdc.decode_summary(out[2])
    assert summ["diverged"] == 1 and summ["no_majority"] == 0 and summ["suspect_mask"] == 0b110
