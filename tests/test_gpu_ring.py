"""GPU ring replay audit (table compare + localize) versus the oracle, the
pages' fault scenarios on device, and the audit table built from per-parameter
gradient fingerprints."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests.test_oracle_ring import scenario_table

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _run(sdc, table_np, offset):
    t = torch.from_numpy(np.ascontiguousarray(table_np).view(np.int64)).to(DEV)
    mism, hits, cul, amb, summ = sdc.ring_audit(t, offset)
    res = sdc.ring_result(mism, cul, offset % max(1, table_np.shape[0]))
    res["hits"] = hits.cpu().tolist()
    res["amb_flags"] = amb.cpu().tolist()
    res["summary"] = np.frombuffer(summ.cpu().numpy().tobytes(), dtype=sdc.RING_SUMMARY_DTYPE)[0]
    return res


def _check(sdc, table_np, offset):
    n = table_np.shape[0]
    got = _run(sdc, table_np, offset)
    tab = [[list(map(int, table_np[r, 0])), list(map(int, table_np[r, 1]))] for r in range(n)]
    pairs = oracle.ring_pairs(tab, offset % n if n else 0)
    culprits, ambiguous = oracle.localize(pairs)
    assert got["pairs"] == pairs
    assert got["culprits"] == culprits
    assert got["ambiguous"] == ambiguous
    hits = [0] * n
    for p in pairs:
        for x in p:
            hits[x] += 1
    assert got["hits"] == hits
    assert int(got["summary"]["n_pairs"]) == len(pairs)
    assert int(got["summary"]["n_culprits"]) == len(culprits)
    assert int(got["summary"]["n_ambiguous"]) == len(ambiguous)


def test_pages_fault_scenarios_on_device(sdc):
    g = json.load(open(os.path.join(GOLDEN, "ring_audit_scenarios.json")))
    for sc in g["scenarios"]:
        tab = np.array(scenario_table(sc["n"], sc["offset"], set(sc["wrong_own"]), set(sc["wrong_replay"])),
                       dtype=np.uint64)
        got = _run(sdc, tab, sc["offset"])
        assert [list(p) for p in got["pairs"]] == sc["printed_pairs"], sc["name"]
        assert got["culprits"] == sc["printed_culprits"], sc["name"]
        _check(sdc, tab, sc["offset"])


@pytest.mark.parametrize("n,L", [(1, 1), (2, 3), (3, 1), (24, 65), (32, 591), (1000, 3), (4097, 33)])
def test_random_tables(sdc, n, L):
    rng = np.random.default_rng(n * 7 + L)
    for trial in range(3):
        offset = int(rng.integers(0, 2 * n + 1))
        base = rng.integers(0, 2 ** 63, size=(n, L), dtype=np.uint64)
        tab = np.empty((n, 2, L), dtype=np.uint64)
        tab[:, 0] = base
        tab[:, 1] = base[(np.arange(n) + offset) % n]
        for _ in range(int(rng.integers(0, max(2, n // 10)))):
            r, row, w = int(rng.integers(n)), int(rng.integers(2)), int(rng.integers(L))
            tab[r, row, w] ^= np.uint64(1 << int(rng.integers(64)))
        _check(sdc, tab, offset)


def test_empty_ring(sdc):
    _check(sdc, np.zeros((0, 2, 4), dtype=np.uint64), 3)


def test_audit_table_from_gradient_fingerprints(sdc):
    """n ranks' own gradients and their replays of their targets, fingerprinted per
    parameter; a persistent fault on one rank is named as the culprit."""
    n, offset = 8, 3
    shapes = [((64, 48), torch.bfloat16), ((48,), torch.float32), ((4096,), torch.bfloat16), ((7, 9), torch.float32)]
    gen = W.generator(77, DEV)
    grads = [[W.normal(s, 1e-3, dt, gen, DEV) for s, dt in shapes] for _ in range(n)]  # rank r's micro-batch
    loss = torch.arange(n, dtype=torch.float32, device=DEV) * 0.25 + 2.0
    replays = [[t.clone() for t in grads[(r + offset) % n]] for r in range(n)]
    bad = 5  # persistent fault: corrupts rank 5's own gradient and the replay it runs
    W.xor_element(grads[bad][2], 100, 1 << 3)
    W.xor_element(replays[bad][0], 7, 1 << 12)
    own_fp = sdc.Plan(grads).fingerprint()      # [n, T, 2]
    rep_fp = sdc.Plan(replays).fingerprint()    # [n, T, 2]
    loss_bits = loss.view(torch.int32).to(torch.int64)
    rep_loss_bits = loss_bits[(torch.arange(n, device=DEV) + offset) % n]
    own_row = torch.cat([loss_bits[:, None], own_fp.reshape(n, -1)], dim=1)
    rep_row = torch.cat([rep_loss_bits[:, None], rep_fp.reshape(n, -1)], dim=1)
    table = torch.stack([own_row, rep_row], dim=1).contiguous()  # [n, 2, 1 + 2T]
    mism, hits, cul, amb, summ = sdc.ring_audit(table, offset)
    res = sdc.ring_result(mism, cul, offset)
    replayer_of_bad = (bad - offset) % n
    assert res["pairs"] == sorted([(bad, replayer_of_bad), ((bad + offset) % n, bad)], key=lambda p: p[1])
    assert res["culprits"] == [bad] and res["ambiguous"] == []
    # the gradient fingerprints themselves agree with the oracle
    from tests._helpers import fp_table, oracle_fp_table
    assert fp_table(own_fp) == oracle_fp_table(grads)
