"""Pins of the oracle's ring audit against the pages' fault-scenario table.

Source: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" -- "Check 2: Ring replay, before the optimizer step" and
the check-2 rows of the "Fault scenarios" table.
"""
import json
import os

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def scenario_table(n, offset, wrong_own, wrong_replay, L=5):
    """Rows of correct results (value = the micro-batch's rank) with the page's faults applied."""
    def result(mb, bad):
        return [mb * 1000 + i + (7_777_777 if bad else 0) for i in range(L)]
    return [[result(r, r in wrong_own), result((r + offset) % n, r in wrong_replay)] for r in range(n)]


def test_pages_fault_scenarios():
    g = json.load(open(os.path.join(GOLDEN, "ring_audit_scenarios.json")))
    for sc in g["scenarios"]:
        table = scenario_table(sc["n"], sc["offset"], set(sc["wrong_own"]), set(sc["wrong_replay"]))
        pairs = oracle.ring_pairs(table, sc["offset"])
        assert [list(p) for p in pairs] == sc["printed_pairs"], sc["name"]
        culprits, ambiguous = oracle.localize(pairs)
        assert culprits == sc["printed_culprits"], sc["name"]
        if not sc["printed_culprits"]:
            assert ambiguous == pairs  # the page confirms these with a third GPU
            assert (pairs[0][0] + sc["offset"]) % sc["n"] == sc["confirmed_by_third_gpu"]


def test_no_fault_no_pairs_and_self_pair_counts_twice():
    table = scenario_table(16, 4, set(), set())
    assert oracle.ring_pairs(table, 4) == []
    # offset 0: every rank replays itself; a mismatch is the pair (r, r), which counts r twice
    t = [[[1, 2], [1, 3]]]
    pairs = oracle.ring_pairs(t, 0)
    assert pairs == [(0, 0)]
    assert oracle.localize(pairs) == ([0], [])
