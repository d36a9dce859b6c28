"""Pins of the oracle's attention invariant.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method section 3: in the attention
backward dV = P^T dO, and every row of the softmax P sums to 1, so
1^T dV = 1^T dO; P is rebuilt in the backward from Q K^T, the softmax and the
log-sum-exp saved by the forward, so an upstream error that breaks the row sums
breaks the invariant too.

Pins: pure-Python loops with math.exp for P and dV, the invariant's identity,
closed forms for a shifted log-sum-exp and for the causal mask's first and last
rows, and an emulation of the kernel's arithmetic (float32 scores, bf16 P,
float32 accumulation rounding to nearest or truncating) that the bound must
cover, with a case that drives the residual to a sizeable share of it.
"""
import math

import numpy as np
import pytest

import oracle


def _bf16_round(x: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _inputs(L, D, seed, causal):
    rng = np.random.default_rng(seed)
    Qb = _bf16_round(rng.standard_normal((L, D)).astype(np.float32))
    Kb = _bf16_round(rng.standard_normal((L, D)).astype(np.float32))
    dOb = _bf16_round(rng.standard_normal((L, D)).astype(np.float32))
    scale = 1.0 / math.sqrt(D)
    Q, K = oracle.bf16_to_f64(Qb), oracle.bf16_to_f64(Kb)
    sc = float(np.float32(scale))
    lse = np.empty(L)
    for i in range(L):  # the forward's log-sum-exp, with math.fsum, row by row
        row = [sc * float(np.dot(Q[i], K[j])) for j in range(L) if not (causal and j > i)]
        m = max(row)
        lse[i] = m + math.log(math.fsum(math.exp(v - m) for v in row))
    return Qb, Kb, dOb, scale, lse


@pytest.mark.parametrize("causal", [False, True])
def test_probs_and_dv_match_python_loops(causal):
    L, D = 6, 3
    Qb, Kb, dOb, scale, lse = _inputs(L, D, 1, causal)
    Q, K, dO = (oracle.bf16_to_f64(x) for x in (Qb, Kb, dOb))
    sc = float(np.float32(scale))
    P = oracle.attn_probs(Qb, Kb, lse, scale, causal)
    for i in range(L):
        for j in range(L):
            s = sum(Q[i, d] * K[j, d] for d in range(D))
            ref = 0.0 if causal and j > i else math.exp(sc * s - lse[i])
            assert abs(P[i, j] - ref) <= 1e-15 * max(1.0, ref)
        assert abs(P[i].sum() - 1.0) < 1e-14  # the forward's log-sum-exp normalises every row
    dV = oracle.attn_dv(P, dOb)
    for j in range(L):
        for c in range(D):
            ref = math.fsum(P[i, j] * dO[i, c] for i in range(L))
            assert abs(dV[j, c] - ref) <= 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_invariant_identity(causal):
    L, D = 48, 16
    Qb, Kb, dOb, scale, lse = _inputs(L, D, 2, causal)
    dV = oracle.attn_dv(oracle.attn_probs(Qb, Kb, lse, scale, causal), dOb)
    v = oracle.attn_invariant(dV.sum(axis=0), dOb)
    assert np.all(np.abs(v["residual"]) <= 1e-12 * np.abs(oracle.bf16_to_f64(dOb)).sum(axis=0))
    assert v["n_flagged"] == 0


def test_causal_first_and_last_rows():
    # query 0 attends key 0 alone (P[0, 0] = 1); key L-1 is attended by query L-1 alone
    L, D = 10, 4
    Qb, Kb, dOb, scale, lse = _inputs(L, D, 3, True)
    P = oracle.attn_probs(Qb, Kb, lse, scale, True)
    assert abs(P[0, 0] - 1.0) < 1e-15 and np.all(P[0, 1:] == 0)
    dV = oracle.attn_dv(P, dOb)
    np.testing.assert_allclose(dV[L - 1], P[L - 1, L - 1] * oracle.bf16_to_f64(dOb)[L - 1], rtol=1e-15)


@pytest.mark.parametrize("delta", [-3.0, 0.5, 4.0])
def test_shifted_lse_closed_form(delta):
    # an upstream error in row i's log-sum-exp scales that row of P by e^-delta: the
    # residual is (e^-delta - 1) dO[i, :] exactly, on every column
    L, D, i = 32, 8, 7
    Qb, Kb, dOb, scale, lse = _inputs(L, D, 4, False)
    bad = lse.copy()
    bad[i] += delta
    dV = oracle.attn_dv(oracle.attn_probs(Qb, Kb, bad, scale, False), dOb)
    v = oracle.attn_invariant(dV.sum(axis=0), dOb)
    expect = (math.exp(-delta) - 1.0) * oracle.bf16_to_f64(dOb)[i]
    np.testing.assert_allclose(v["residual"], expect, rtol=1e-9, atol=1e-12)


def _emulate(Qb, Kb, dOb, lse, scale, causal, mode):
    """The kernel's arithmetic: float32 scores (round to nearest per step), P in
    float32 then bf16, dV accumulated in float32 over the query rows in order."""
    Q, K, dO = (oracle.bf16_to_f64(x) for x in (Qb, Kb, dOb))
    L, D = Q.shape
    S = np.zeros((L, L))
    for d in range(D):
        S = (S + np.outer(Q[:, d], K[:, d])).astype(np.float32).astype(np.float64)
    arg = (S * float(np.float32(scale)) - np.asarray(lse, np.float32)[:, None]).astype(np.float32)
    P = oracle.bf16_to_f64(_bf16_round(np.exp(arg.astype(np.float64)).astype(np.float32)))
    if causal:
        P = np.tril(P)
    acc = np.zeros((L, dO.shape[1]))
    for i in range(L):
        x = acc + np.outer(P[i], dO[i])
        r = x.astype(np.float32).astype(np.float64)
        if mode == "trunc":
            over = np.abs(r) > np.abs(x)
            r[over] = np.nextafter(r[over].astype(np.float32), np.float32(0)).astype(np.float64)
        acc = r
    return acc


@pytest.mark.parametrize("mode", ["rn", "trunc"])
@pytest.mark.parametrize("causal", [False, True])
def test_bound_covers_kernel_arithmetic(mode, causal):
    L, D = 96, 32
    Qb, Kb, dOb, scale, lse = _inputs(L, D, 5, causal)
    acc = _emulate(Qb, Kb, dOb, np.float32(lse), scale, causal, mode)
    v = oracle.attn_invariant(acc.sum(axis=0), dOb)
    assert v["n_flagged"] == 0
    assert np.max(np.abs(v["residual"]) / v["bound"]) <= 1.0


def test_bound_not_vacuous():
    # zero scores: every P is 1/L rounded to bf16 with one sign of error for L = 96,
    # all-positive dO: the row-sum error adds up on every column
    L, D = 96, 8
    Qb = np.zeros((L, D), np.uint16)
    Kb = np.zeros((L, D), np.uint16)
    dOb = _bf16_round(np.random.default_rng(6).uniform(0.5, 1.0, (L, D)).astype(np.float32))
    lse = np.full(L, math.log(L))
    acc = _emulate(Qb, Kb, dOb, np.float32(lse), 1.0, False, "rn")
    v = oracle.attn_invariant(acc.sum(axis=0), dOb)
    ratio = np.abs(v["residual"]) / v["bound"]
    assert v["n_flagged"] == 0 and ratio.max() <= 1.0
    assert ratio.min() > 0.1


def test_flag_rule_edges():
    L, D = 4, 3
    dOb = np.zeros((L, D), np.uint16)
    b = 2.0 ** -100
    v = oracle.attn_invariant(np.array([b, 2 * b, np.nan]), dOb)
    assert list(v["flag"]) == [0, 1, 1]


@pytest.mark.parametrize("causal", [False, True])
def test_probs_of_a_key_block_are_columns_of_the_full_matrix(causal):
    # a block of keys key0 .. key0 + n - 1 gives exactly those columns of P, causal mask included
    L, D = 40, 8
    Qb, Kb, dOb, scale, lse = _inputs(L, D, 7, causal)
    P = oracle.attn_probs(Qb, Kb, lse, scale, causal)
    for key0, n in [(0, 8), (13, 9), (32, 8)]:
        Pb = oracle.attn_probs(Qb, Kb[key0:key0 + n], lse, scale, causal, key0=key0)
        np.testing.assert_allclose(Pb, P[:, key0:key0 + n], rtol=1e-13, atol=0)
        np.testing.assert_array_equal(Pb == 0, P[:, key0:key0 + n] == 0)
        if causal:
            assert np.all(Pb[:key0] == 0)  # no query before the block attends any of its keys
