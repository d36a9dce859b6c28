"""Pins of the oracle's strict-majority vote.

Source: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" -- "Check 3: Weight fingerprints, after the optimizer step"
and "Beyond DDP".
"""
import itertools
import json
import os

import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_page_rule_cases():
    g = json.load(open(os.path.join(GOLDEN, "vote_rules.json")))
    for case in g["cases"]:
        table = [[(ord(c), 0)] for c in case["copies"]]
        _, _, summ = oracle.vote(table)
        assert oracle.pages_verdict(summ) == {"diverged": case["diverged"], "suspects": case["suspects"]}


def _majority_by_sorting(copies):
    """Strict-majority element found another way: after sorting, a value held by
    more than half of the copies must sit in the middle position."""
    s = sorted(copies)
    mid = s[len(s) // 2]
    return mid if 2 * copies.count(mid) > len(copies) else None


@pytest.mark.parametrize("R", [2, 3, 4, 5, 6])
def test_brute_force_all_tuples(R):
    for tup in itertools.product("abc", repeat=R):
        table = [[(ord(c), 1)] for c in tup]
        suspect, mask, summ = oracle.vote(table)
        if len(set(tup)) == 1:
            assert suspect == [-1] and mask == [0] and summ["diverged"] == 0
            continue
        maj = _majority_by_sorting(list(tup))
        assert summ["diverged"] == 1
        if maj is None:
            assert suspect == [-3] and mask == [0] and summ["no_majority"] == 1
        else:
            odd = [r for r, c in enumerate(tup) if c != maj]
            assert mask == [sum(1 << r for r in odd)]
            assert suspect == [odd[0] if len(odd) == 1 else -2]
            assert oracle.pages_verdict(summ) == {"diverged": True, "suspects": odd}


def test_permutation_equivariance():
    base = [(1, 1), (1, 1), (2, 2), (1, 1), (3, 3)]
    ref_mask = oracle.vote([[c] for c in base])[1][0]
    for perm in itertools.permutations(range(5)):
        table = [[base[perm[r]]] for r in range(5)]
        m = oracle.vote(table)[1][0]
        assert m == sum(1 << r for r in range(5) if (ref_mask >> perm[r]) & 1)


def test_no_majority_anywhere_hides_named_suspects():
    # tensor 0 names replica 2, tensor 1 has no strict majority: the page returns None
    table = [[(0, 0), (5, 5)], [(0, 0), (5, 5)], [(9, 9), (6, 6)], [(0, 0), (6, 6)]]
    suspect, mask, summ = oracle.vote(table)
    assert suspect == [2, -3] and mask == [4, 0]
    assert oracle.pages_verdict(summ) == {"diverged": True, "suspects": None}
    assert summ["suspect_mask"] == 4


def test_first_element_differs_only_in_weighted_sum():
    table = [[(7, 1)], [(7, 2)], [(7, 1)]]
    assert oracle.vote(table)[0] == [1]
