"""GPU vote parity with the oracle's vote, and the fingerprint -> vote pipeline."""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import fp_table

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _run_vote(sdc, table_np):
    fp = torch.from_numpy(table_np.view(np.int64)).to(DEV)
    suspect, mask, summary = sdc.vote(fp)
    return (suspect.cpu().tolist(), [int(m) & ((1 << 64) - 1) for m in mask.cpu().numpy().view(np.uint64)],
            sdc.decode_summary(summary))


def _oracle(table_np):
    R, T = table_np.shape[:2]
    tab = [[(int(table_np[r, k, 0]), int(table_np[r, k, 1])) for k in range(T)] for r in range(R)]
    return oracle.vote(tab)


def _check(sdc, table_np):
    s, m, summ = _run_vote(sdc, table_np)
    rs, rm, rsumm = _oracle(table_np)
    assert s == rs and m == rm
    for key in ("diverged", "no_majority", "suspect_mask"):
        assert summ[key] == rsumm[key], key
    assert sdc.pages_verdict(summ) == oracle.pages_verdict(rsumm)


def test_golden_rule_cases(sdc):
    g = json.load(open(os.path.join(GOLDEN, "vote_rules.json")))
    for case in g["cases"]:
        R = len(case["copies"])
        t = np.zeros((R, 1, 2), dtype=np.uint64)
        for r, c in enumerate(case["copies"]):
            t[r, 0, 0] = ord(c)
        _, _, summ = _run_vote(sdc, t)
        assert sdc.pages_verdict(summ) == {"diverged": case["diverged"], "suspects": case["suspects"]}


@pytest.mark.parametrize("R", [1, 2, 3, 4, 5, 6])
def test_every_tuple_over_three_values(sdc, R):
    tuples = list(itertools.product(range(3), repeat=R))
    t = np.zeros((R, len(tuples), 2), dtype=np.uint64)
    for k, tup in enumerate(tuples):
        for r, v in enumerate(tup):
            t[r, k, 0] = 1000 + v
            t[r, k, 1] = v  # differ in both sums
    s, m, summ = _run_vote(sdc, t)
    rs, rm, rsumm = _oracle(t)
    assert s == rs and m == rm and summ["suspect_mask"] == rsumm["suspect_mask"]
    assert summ["n_differing"] == sum(1 for tup in tuples if len(set(tup)) > 1)


@pytest.mark.parametrize("R,T", [(3, 1), (8, 291), (3, 100_000), (64, 500), (63, 7)])
def test_random_tables(sdc, R, T):
    rng = np.random.default_rng(R * 1000 + T)
    base = rng.integers(0, 2 ** 63, size=(T, 2), dtype=np.uint64)
    t = np.repeat(base[None], R, axis=0).copy()
    for _ in range(max(1, T // 20)):  # corrupt random copies, sometimes only W
        r, k = int(rng.integers(R)), int(rng.integers(T))
        t[r, k, int(rng.integers(2))] ^= np.uint64(1 << int(rng.integers(64)))
    # a few tensors with no strict majority
    if R >= 2 and T > 3:
        for r in range(R // 2 + 1):
            t[r, 3, 0] ^= np.uint64(r + 1)
    _check(sdc, t)


def test_empty_and_uniform(sdc):
    _check(sdc, np.zeros((4, 0, 2), dtype=np.uint64))
    _check(sdc, np.ones((5, 10, 2), dtype=np.uint64))


def test_pipeline_names_injected_replica(sdc):
    w = W.tiny(DEV, seed=3)
    plan = sdc.Plan(w["replicas"])
    fp = plan.fingerprint()
    suspect, mask, summary = sdc.vote(fp)
    k = w["truth"]["tensor"]
    exp = [-1] * len(W.TINY_SHAPES)
    exp[k] = 1
    assert suspect.cpu().tolist() == exp
    assert sdc.pages_verdict(sdc.decode_summary(summary)) == {"diverged": True, "suspects": [1]}


def test_worked_example_on_device(sdc):
    """The page's example: identical updates leave identical fingerprints (fault or not)."""
    for fault in (False, True):
        ex = W.worked_example(DEV, fault=fault)
        avg, pre, post = sdc.grad_average_scan(ex["grads"])
        weights = [w - ex["lr"] * avg for w in ex["weights"]]
        plan = sdc.Plan([[w] for w in weights])
        _, _, summary = sdc.vote(plan.fingerprint())
        assert sdc.pages_verdict(sdc.decode_summary(summary)) == {"diverged": False, "suspects": []}
        assert round(float(weights[0]), 3) == (0.350 if fault else 0.470)
        ref = oracle.average([np.array([float(g)], dtype=np.float32) for g in ex["grads"]], "f32")
        assert int(avg.view(torch.int32).cpu()[0]) & 0xFFFFFFFF == int(ref[0])
