"""The data-parallel classes on one GPU, through the C ABI's kernels.

With one rank (no process group) the gathered table is the local one.  The
test checks:
- WeightCheck: its table against the oracle's fingerprints, and its verdict
  against the oracle's vote.  ``suspects`` are ranks (here rank 0, which
  holds the odd copy); ``suspect_replicas`` are the copies.
- GradCheck: both halves' statistics against the oracle's, on the bytes the
  buffers hold at each point.
The exchanges between ranks are covered by test_dp_gloo.py (gloo, on the CPU).
"""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import host_bits, stats_match

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def dp():
    from silent_corruption_checksums_gb300 import dp as m
    return m


def _oracle_table(reps):
    return np.array([[oracle.fingerprint(host_bits(t)) for t in ts] for ts in reps], dtype=np.uint64)


@pytest.mark.parametrize("n_copies", [1, 2, 3, 5])
def test_weight_check_one_rank(dp, n_copies):
    w = W.weights_1b(DEV, seed=11, n_replicas=n_copies, n_layers=1)
    reps = w["replicas"]
    wc = dp.WeightCheck(reps)
    res = wc()
    table = wc.table.cpu().numpy().view(np.uint64)
    ref = _oracle_table(reps)
    assert np.array_equal(table, ref)
    verdict = oracle.pages_verdict(oracle.vote(ref.tolist())[2])
    assert {"diverged": res["diverged"], "suspects": res["suspect_replicas"]} == verdict
    if n_copies >= 3:
        assert res["suspects"] == [0] and res["suspect_replicas"] == [w["truth"]["replica"]]
    elif n_copies == 2:
        assert res["suspects"] is None  # two copies: a disagreement, no rank named
    else:
        assert res == {"diverged": False, "suspects": [], "suspect_replicas": []}
    # a second call on the same buffers after repairing the copy agrees everywhere
    if n_copies >= 2:
        k, e, bit = w["truth"]["tensor"], w["truth"]["element"], w["truth"]["bit"]
        W.xor_element(reps[w["truth"]["replica"]][k], e, 1 << bit)
        assert wc() == {"diverged": False, "suspects": [], "suspect_replicas": []}
    wc.close()


def test_grad_check_one_rank(dp):
    g = W.grads_flat(3 * 8192 + 11, 1, torch.bfloat16, 1e-3, DEV, seed=12, inject_buf=0, rate=1e-3)
    grads = [g["bufs"][0][:5000], g["bufs"][0][5000:]]
    gc = dp.GradCheck(grads)
    before = gc.before_allreduce()
    ref = oracle.grad_stats_multi([host_bits(t) for t in grads], ["bf16", "bf16"])
    stats_match(before["stats"][0], ref)
    assert before["nonfinite"] == ([0] if ref["nonfinite_fp32"] else [])
    # the all-reduce of one rank leaves the gradient as it is; a NaN written into it is seen after
    after = gc.after_allreduce()
    stats_match(after["stats"], ref)
    grads[1][7] = float("nan")
    after = gc.after_allreduce()
    stats_match(after["stats"], oracle.grad_stats_multi([host_bits(t) for t in grads], ["bf16", "bf16"]))
    assert after["bad"] is True
    gc.close()
