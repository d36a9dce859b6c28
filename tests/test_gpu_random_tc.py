"""Seeded random sweep of the tensor-core kernels against the oracle: the GEMM
with row (and column) checksums over random tile-aligned shapes and input
scales, and the attention backward's dV half with its invariant over random
head counts, lengths and masks.

Sources: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method sections 2 and 3.
"""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("case", range(8))
def test_gemm_random(sdc, case):
    rng = np.random.default_rng(1000 + case)
    M = 128 * int(rng.integers(1, 9))
    N = 256 * int(rng.integers(1, 7))
    K = 64 * int(rng.integers(1, 33))
    a_std = float(2.0 ** rng.integers(-6, 7))
    w_std = float(2.0 ** rng.integers(-8, 3))
    cols = bool(rng.integers(0, 2))
    ops = W.gemm_operands(M, N, K, DEV, seed=2000 + case, a_std=a_std, w_std=w_std)
    g = sdc.AbftGemm(M, N, K, DEV, columns=cols)
    g(ops["A"], ops["W"])
    torch.cuda.synchronize()
    assert int(g.aborted[0]) == 0
    Ab, Wb = _bits(ops["A"]), _bits(ops["W"])
    exact = oracle.abft_product(Ab, Wb)
    A64, W64 = oracle.bf16_to_f64(Ab), oracle.bf16_to_f64(Wb)
    gk = K * 2.0 ** -22
    e = gk * (1.0 + gk) * (np.abs(A64) @ np.abs(W64).T) + 2.0 * K * 2.0 ** -126
    C = g.C.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(C - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134), (M, N, K)
    v = oracle.abft_verify(g.rowsum.cpu().numpy(), Ab, Wb)
    assert np.all(np.abs(g.rowsum.cpu().numpy() - exact.sum(axis=1)) <= v["bound"])
    assert v["n_flagged"] == 0 and int(g.summary[0]) == 0 and np.all(g.flag.cpu().numpy() == 0)
    if cols:
        vc = oracle.abft_verify_cols(g.colsum.cpu().numpy(), Ab, Wb)
        assert np.all(np.abs(g.colsum.cpu().numpy() - exact.sum(axis=0)) <= vc["bound"])
        assert vc["n_flagged"] == 0 and int(g.summary[1]) == 0 and np.all(g.flag_col.cpu().numpy() == 0)


@pytest.mark.parametrize("case", range(6))
def test_wgrad_random(sdc, case):
    # the weight-gradient form over random shapes (multiples of 8, rarely tile-aligned), token
    # counts from one to a few thousand and random input scales, rows and columns checked
    rng = np.random.default_rng(5000 + case)
    T = int(rng.integers(1, 3000))
    N = 8 * int(rng.integers(1, 100))
    K = 8 * int(rng.integers(1, 100))
    dy_std = float(2.0 ** rng.integers(-16, 0))
    x_std = float(2.0 ** rng.integers(-4, 5))
    ops = W.wgrad_operands(T, N, K, DEV, seed=6000 + case, dy_std=dy_std, x_std=x_std)
    a = sdc.AbftWgrad(T, N, K, DEV)
    a(ops["dY"], ops["X"])
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0
    dYb, Xb = _bits(ops["dY"]), _bits(ops["X"])
    exact = oracle.wgrad_product(dYb, Xb)
    g = T * 2.0 ** -22
    e = g * (1.0 + g) * (np.abs(oracle.bf16_to_f64(dYb)).T @ np.abs(oracle.bf16_to_f64(Xb))) + 2.0 * T * 2.0 ** -126
    dW = a.dW.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(dW - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134), (T, N, K)
    v = oracle.wgrad_verify(a.rowsum.cpu().numpy(), a.colsum.cpu().numpy(), dYb, Xb)
    assert np.all(np.abs(a.rowsum.cpu().numpy() - exact.sum(axis=1)) <= v["bound"])
    assert np.all(np.abs(a.colsum.cpu().numpy() - exact.sum(axis=0)) <= v["bound_col"])
    assert v["n_flagged"] == 0 and v["n_flagged_col"] == 0
    assert int(a.summary[0]) == 0 and int(a.summary[1]) == 0


@pytest.mark.parametrize("case", range(14))
def test_attention_random(sdc, case):
    # heads and lengths drawn so that the (head, key block) items range from one to a few
    # hundred: fewer than, about as many as and several times the persistent grid
    rng = np.random.default_rng(3000 + case)
    BH = int(rng.integers(1, 4)) if case < 6 else int(rng.integers(4, 17))
    L = 128 * int(rng.integers(1, 7)) if case < 6 else 128 * int(rng.integers(4, 17))
    causal = bool(rng.integers(0, 2))
    x = W.attn_inputs(BH, L, DEV, seed=4000 + case, causal=causal)
    a = sdc.AttnDvCheck(BH, L, DEV)
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], causal)
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    Qb, Kb, dOb = _bits(x["Q"]), _bits(x["K"]), _bits(x["dO"])
    lse = x["lse"].cpu().numpy()
    dV = a.dV.float().cpu().numpy().astype(np.float64)
    g = L * 2.0 ** -22
    eps = 2.0 ** -8 * (1 + 2.0 ** -7) + g * (1 + g) * (1 + 2.0 ** -7)
    for h in range(BH):
        P = oracle.attn_probs(Qb[h], Kb[h], lse[h], x["scale"], causal)
        exact = oracle.attn_dv(P, dOb[h])
        e = eps * (P.T @ np.abs(oracle.bf16_to_f64(dOb[h])))
        assert np.all(np.abs(dV[h] - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134), (BH, L, causal)
        v = oracle.attn_invariant(a.colsum_dv[h].cpu().numpy(), dOb[h])
        assert v["n_flagged"] == 0
        assert np.all(np.abs(a.colsum_dv[h].cpu().numpy() - exact.sum(axis=0)) <= v["bound"])
