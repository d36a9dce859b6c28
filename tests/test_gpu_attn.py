"""GPU dV half of the attention backward with the invariant 1^T dV = 1^T dO,
versus the oracle.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method section 3.  dV and dV's column
sums come from the tensor cores' float32 accumulator (its own summation order)
and from bf16 probabilities, so they are compared with the oracle's exact values
within the rounding bound; dO's column sums, the bound and the residual are
compared with the oracle's on the kernel's outputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import ATTN_OWN_SLACK, assert_attn_bound

pytestmark = pytest.mark.gpu
DEV = "cuda"
CASES = [(1, 128, False), (1, 128, True), (2, 256, True), (3, 384, False), (2, 1024, True), (1, 1024, False)]


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _run(sdc, x, tol_scale=1.0):
    BH, L, _ = x["Q"].shape
    a = sdc.AttnDvCheck(BH, L, DEV)
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], x["causal"], tol_scale)
    torch.cuda.synchronize()
    return a


# dO's column sums: float32 chains of eight rows folded into float32 pairs
DO_SLACK = 2.0 ** -40 + 8.0 * 2.0 ** -24


def _absd(dOb: np.ndarray) -> np.ndarray:
    """sum_i |dO[i, c]| for one head's bf16 bits [rows, 128]."""
    return np.abs(oracle.bf16_to_f64(dOb)).sum(axis=0)


def _eps(L):
    g = L * 2.0 ** -22
    rho = 1.0 + 2.0 ** -7
    return 2.0 ** -8 * rho + g * (1.0 + g) * rho


@pytest.mark.parametrize("BH,L,causal", CASES)
def test_dv_and_invariant_parity(sdc, BH, L, causal):
    x = W.attn_inputs(BH, L, DEV, seed=BH * 1000 + L + causal, causal=causal)
    a = _run(sdc, x)
    assert int(a.aborted[0]) == 0
    Qb, Kb, dOb = _bits(x["Q"]), _bits(x["K"]), _bits(x["dO"])
    lse = x["lse"].cpu().numpy()
    dV = a.dV.float().cpu().numpy().astype(np.float64)
    eps = _eps(L)
    for h in range(BH):
        P = oracle.attn_probs(Qb[h], Kb[h], lse[h], x["scale"], causal)
        exact = oracle.attn_dv(P, dOb[h])
        mag = P.T @ np.abs(oracle.bf16_to_f64(dOb[h]))  # sum_i P[i, j] |dO[i, c]|
        # each probability within 2^-8 of itself, each accumulation step within two ulps,
        # then the bf16 rounding of dV (2^-8 of the value, 2^-134 if subnormal)
        e = eps * mag
        tol = 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134
        assert np.all(np.abs(dV[h] - exact) <= tol), np.max(np.abs(dV[h] - exact) / tol)
        # dV's column sums from the accumulator: within the bound of the exact column sums
        v = oracle.attn_invariant(a.colsum_dv[h].cpu().numpy(), dOb[h])
        cs = a.colsum_dv[h].cpu().numpy()
        assert np.all(np.abs(cs - exact.sum(axis=0)) <= v["bound"])
        # dO's column sums (float32 pairs), the bound and the residual against the oracle's
        dO = oracle.bf16_to_f64(dOb[h])
        absd = np.abs(dO).sum(axis=0)
        assert np.all(np.abs(a.colsum_do[h].cpu().numpy() - dO.sum(axis=0)) <= DO_SLACK * absd)
        assert_attn_bound(a.bound[h].cpu().numpy(), v["bound"], _absd(dOb[h]))
        assert np.all(np.abs(a.residual[h].cpu().numpy() - v["residual"]) <= ATTN_OWN_SLACK * absd)
        assert v["n_flagged"] == 0 and np.all(a.flag[h].cpu().numpy() == 0)
        assert float(np.max(np.abs(v["residual"]) / v["bound"])) < 0.5
    assert int(a.summary[0]) == 0


def test_deterministic(sdc):
    x = W.attn_inputs(2, 512, DEV, seed=31, causal=True)
    a = _run(sdc, x)
    dV0, cs0 = a.dV.clone(), a.colsum_dv.clone()
    for _ in range(3):
        a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], x["causal"])
        assert torch.equal(a.dV, dV0)
        assert torch.equal(a.colsum_dv.view(torch.int64), cs0.view(torch.int64))


def _expected_flags(x, Kb_used, lse_used, h):
    """Oracle residuals of the faulty run: P from the inputs the kernel saw, the check's
    right-hand side from the clean dO; a column is 'clear' when its exact residual is
    beyond twice the bound, 'clean' when it is inside a tenth of it."""
    Qb, dOb = _bits(x["Q"]), _bits(x["dO"])
    with np.errstate(over="ignore", invalid="ignore"):
        P = oracle.attn_probs(Qb[h], Kb_used[h], lse_used[h], x["scale"], x["causal"])
        v = oracle.attn_invariant(oracle.attn_dv(P, dOb[h]).sum(axis=0), dOb[h])
    r = np.abs(v["residual"])
    return (r > 2.0 * v["bound"]) | np.isnan(r), r < 0.1 * v["bound"]


@pytest.mark.parametrize("delta", [-3.0, 2.0])
def test_shifted_lse_row_flags(sdc, delta):
    # an upstream error in one row's softmax statistics: the row of P no longer sums to 1
    x = W.attn_inputs(2, 256, DEV, seed=32, causal=False)
    h, i = 1, 77
    bad = x["lse"].clone()
    bad[h, i] += delta
    a = _run(sdc, dict(x, lse=bad))
    assert int(a.aborted[0]) == 0
    assert np.all(a.flag[0].cpu().numpy() == 0)  # the other head is untouched
    clear, clean = _expected_flags(x, _bits(x["K"]), bad.cpu().numpy(), h)
    flag = a.flag[h].cpu().numpy()
    assert np.all(flag[clear] == 1) and np.all(flag[clean] == 0)
    if delta < 0:  # |(e^3 - 1) dO[i, c]| clears 2^-8 sum_i |dO[i, c]| on most columns
        assert int(clear.sum()) >= 40
    else:  # (e^-2 - 1) dO[i, c] is within the bf16 noise floor on most columns: a few clear it
        assert int(clear.sum()) >= 1
    assert int(a.summary[0]) == int(a.flag.sum())


def test_corrupted_key_flags(sdc):
    # an upstream error in K (one element's top exponent bit): its column of scores
    # changes for every query while the forward's log-sum-exp stays the clean one
    x = W.attn_inputs(1, 384, DEV, seed=33, causal=True)
    Kf = x["K"].clone()
    W.xor_element(Kf, 5 * 128 + 17, 0x4000)
    a = _run(sdc, dict(x, K=Kf))
    assert int(a.aborted[0]) == 0
    clear, clean = _expected_flags(x, _bits(Kf), x["lse"].cpu().numpy(), 0)
    flag = a.flag[0].cpu().numpy()
    assert np.all(flag[clear] == 1) and np.all(flag[clean] == 0)


def test_rejects_bad_arguments(sdc):
    x = W.attn_inputs(1, 128, DEV, seed=34, causal=False)
    a = sdc.AttnDvCheck(1, 128, DEV)
    args = [x["Q"].data_ptr(), x["K"].data_ptr(), x["dO"].data_ptr(), x["lse"].data_ptr(), 1, 128, 128,
            x["scale"], 0, 1.0, a.dV.data_ptr(), a.colsum_dv.data_ptr(), a.colsum_do.data_ptr(),
            a.residual.data_ptr(), a.bound.data_ptr(), a.flag.data_ptr(), a.summary.data_ptr(),
            a.aborted.data_ptr(), a.ws.data_ptr(), a.ws_bytes, 0]
    for i, v, status in [(6, 64, 9), (5, 102, 9), (7, math.nan, 9), (8, 2, 9), (19, a.ws_bytes - 256, 5),
                         (0, x["Q"].data_ptr() + 2, 8)]:
        bad = list(args)
        bad[i] = v
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_attn_dv_check(*bad)
        assert ei.value.status == status, (i, v)


def _check_against_oracle(sdc, x, a, causal):
    BH = x["Q"].shape[0]
    Qb, Kb, dOb = _bits(x["Q"]), _bits(x["K"]), _bits(x["dO"])
    lse = x["lse"].cpu().numpy()
    dV = a.dV.float().cpu().numpy().astype(np.float64)
    eps = _eps(x["Q"].shape[1])
    for h in range(BH):
        P = oracle.attn_probs(Qb[h], Kb[h], lse[h], x["scale"], causal)
        exact = oracle.attn_dv(P, dOb[h])
        e = eps * (P.T @ np.abs(oracle.bf16_to_f64(dOb[h])))
        assert np.all(np.abs(dV[h] - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134), h
        v = oracle.attn_invariant(a.colsum_dv[h].cpu().numpy(), dOb[h])
        assert np.all(np.abs(a.colsum_dv[h].cpu().numpy() - exact.sum(axis=0)) <= v["bound"]), h
        assert_attn_bound(a.bound[h].cpu().numpy(), v["bound"], _absd(dOb[h]))
        assert v["n_flagged"] == 0 and np.all(a.flag[h].cpu().numpy() == 0), h


@pytest.mark.parametrize("BH,L", [(151, 128), (152, 128), (153, 128), (1, 2048)])
def test_work_items_around_the_grid(sdc, BH, L):
    # (head, key block) items one fewer than, equal to and one more than the persistent grid
    # (one block per SM on this GPU), and one head split over sixteen items
    x = W.attn_inputs(BH, L, DEV, seed=35 + BH, causal=True)
    a = _run(sdc, x)
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    _check_against_oracle(sdc, x, a, True)


def test_counters_reset_between_calls(sdc):
    # the same object (workspace, counters) called causal, non-causal, causal again
    xc = W.attn_inputs(3, 512, DEV, seed=36, causal=True)
    xn = W.attn_inputs(3, 512, DEV, seed=37, causal=False)
    a = sdc.AttnDvCheck(3, 512, DEV)
    for x, causal in [(xc, True), (xn, False), (xc, True)]:
        a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], causal)
        torch.cuda.synchronize()
        assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
        _check_against_oracle(sdc, x, a, causal)


def test_long_sequence_sampled_keys(sdc):
    # one head of 65,536 tokens, causal: 512 key blocks of up to 512 query steps; four key
    # blocks (first, second, middle, last) against the oracle row by row, and the invariant of
    # every column (the kernel's column sums of dV against the oracle's bound)
    L = 1 << 16
    x = W.attn_inputs(1, L, DEV, seed=38, causal=True)
    a = _run(sdc, x)
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    Qb, Kb, dOb = _bits(x["Q"])[0], _bits(x["K"])[0], _bits(x["dO"])[0]
    lse = x["lse"][0].cpu().numpy()
    absdo = np.abs(oracle.bf16_to_f64(dOb))
    eps = _eps(L)
    dV = a.dV[0].float().cpu().numpy().astype(np.float64)
    for j0 in (0, 128, L // 2, L - 128):
        P = oracle.attn_probs(Qb, Kb[j0:j0 + 128], lse, x["scale"], True, key0=j0)  # [L, 128]
        exact = oracle.attn_dv(P, dOb)
        e = eps * (P.T @ absdo)
        tol = 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134
        assert np.all(np.abs(dV[j0:j0 + 128] - exact) <= tol), j0
    v = oracle.attn_invariant(a.colsum_dv[0].cpu().numpy(), dOb)
    assert v["n_flagged"] == 0 and np.all(a.flag[0].cpu().numpy() == 0)
    assert_attn_bound(a.bound[0].cpu().numpy(), v["bound"], _absd(dOb))


@pytest.mark.parametrize("BH,group,L,causal", [(8, 4, 512, True), (8, 4, 384, False), (6, 2, 256, True),
                                               (8, 8, 256, True)])
def test_grouped_query_attention(sdc, BH, group, L, causal):
    # group query heads per K/V head (4: the 8b layout's 32 query heads over 8 K/V heads; 8: one
    # K/V head): dV of a K/V head sums P_h^T dO_h over its group, and its column sums equal the
    # group's column sums of dO; the oracle stacks the group's rows of P and of dO
    x = W.attn_inputs(BH, L, DEV, seed=60 + BH + group + L, causal=causal, group=group)
    a = sdc.AttnDvCheck(BH, L, DEV, group=group)
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], causal)
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    Qb, Kb, dOb = _bits(x["Q"]), _bits(x["K"]), _bits(x["dO"])
    lse = x["lse"].cpu().numpy()
    dV = a.dV.float().cpu().numpy().astype(np.float64)
    eps = _eps(group * L)
    for v in range(BH // group):
        heads = range(v * group, (v + 1) * group)
        P = np.vstack([oracle.attn_probs(Qb[h], Kb[v], lse[h], x["scale"], causal) for h in heads])
        dOs = np.vstack([dOb[h] for h in heads])
        exact = oracle.attn_dv(P, dOs)
        e = eps * (P.T @ np.abs(oracle.bf16_to_f64(dOs)))
        assert np.all(np.abs(dV[v] - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134), v
        inv = oracle.attn_invariant(a.colsum_dv[v].cpu().numpy(), dOs)
        assert np.all(np.abs(a.colsum_dv[v].cpu().numpy() - exact.sum(axis=0)) <= inv["bound"]), v
        assert_attn_bound(a.bound[v].cpu().numpy(), inv["bound"], _absd(dOs))
        absd = np.abs(oracle.bf16_to_f64(dOs)).sum(axis=0)
        assert np.all(np.abs(a.colsum_do[v].cpu().numpy() - oracle.bf16_to_f64(dOs).sum(axis=0)) <= DO_SLACK * absd)
        assert inv["n_flagged"] == 0 and np.all(a.flag[v].cpu().numpy() == 0), v


def test_grouped_rejects_bad_shapes(sdc):
    with pytest.raises(ValueError):
        sdc.AttnDvCheck(6, 128, DEV, group=4)
    x = W.attn_inputs(4, 128, DEV, seed=64, causal=True, group=2)
    a = sdc.AttnDvCheck(4, 128, DEV, group=2)
    with pytest.raises(ValueError):  # K of every query head where the group's K/V heads are expected
        a(x["Q"], x["Q"], x["dO"], x["lse"], x["scale"], True)


@pytest.mark.parametrize("BH,group,L,causal", [(2, 1, 100, True), (1, 1, 260, False), (3, 1, 1000, True),
                                               (8, 4, 300, True), (1, 1, 4100, False), (2, 2, 4, True)])
def test_ragged_lengths(sdc, BH, group, L, causal):
    # sequence lengths that are not multiples of the 128-token blocks (any multiple of 4): the last
    # key block and the last query block are partial; the copies read zeros past L inside each
    # head, and keys and queries past L take no probability
    x = W.attn_inputs(BH, L, DEV, seed=90 + BH + L, causal=causal, group=group)
    a = sdc.AttnDvCheck(BH, L, DEV, group=group)
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], causal)
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    Qb, Kb, dOb = _bits(x["Q"]), _bits(x["K"]), _bits(x["dO"])
    lse = x["lse"].cpu().numpy()
    dV = a.dV.float().cpu().numpy().astype(np.float64)
    eps = _eps(group * L)
    for v in range(BH // group):
        heads = range(v * group, (v + 1) * group)
        P = np.vstack([oracle.attn_probs(Qb[h], Kb[v], lse[h], x["scale"], causal) for h in heads])
        dOs = np.vstack([dOb[h] for h in heads])
        exact = oracle.attn_dv(P, dOs)
        e = eps * (P.T @ np.abs(oracle.bf16_to_f64(dOs)))
        assert np.all(np.abs(dV[v] - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134), v
        inv = oracle.attn_invariant(a.colsum_dv[v].cpu().numpy(), dOs)
        assert np.all(np.abs(a.colsum_dv[v].cpu().numpy() - exact.sum(axis=0)) <= inv["bound"]), v
        assert_attn_bound(a.bound[v].cpu().numpy(), inv["bound"], _absd(dOs))
        assert inv["n_flagged"] == 0 and np.all(a.flag[v].cpu().numpy() == 0), v


def test_length_not_a_multiple_of_4_is_rejected(sdc):
    x = W.attn_inputs(1, 128, DEV, seed=95, causal=True)
    a = sdc.AttnDvCheck(1, 128, DEV)
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_attn_dv_check(x["Q"].data_ptr(), x["K"].data_ptr(), x["dO"].data_ptr(), x["lse"].data_ptr(), 1, 126,
                              128, x["scale"], 1, 1.0, a.dV.data_ptr(), a.colsum_dv.data_ptr(), a.colsum_do.data_ptr(),
                              a.residual.data_ptr(), a.bound.data_ptr(), a.flag.data_ptr(), a.summary.data_ptr(),
                              a.aborted.data_ptr(), a.ws.data_ptr(), a.ws_bytes, 0)
    assert ei.value.status == 9


@pytest.mark.parametrize("BH,L,causal", [(64, 2048, False), (40, 2052, True)])
def test_prep_pass_several_blocks_per_cta(sdc, BH, L, causal):
    # more (head, 128-row block) units than the prep pass's persistent CTAs (three per SM), so
    # each CTA sums several blocks through its two alternating buffers; dO's column sums and the
    # bound of every head against exact sums, dV's column sums within that bound
    x = W.attn_inputs(BH, L, DEV, seed=39, causal=causal)
    a = _run(sdc, x)
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    dO = oracle.bf16_to_f64(_bits(x["dO"]))  # [BH, L, 128]
    colsum_do = a.colsum_do.cpu().numpy()
    absd = np.abs(dO).sum(axis=1)
    assert np.all(np.abs(colsum_do - dO.sum(axis=1)) <= DO_SLACK * absd)
    assert_attn_bound(a.bound.cpu().numpy(), oracle.attn_bound(absd, L), absd)
    assert np.all(np.abs(a.residual.cpu().numpy()) <= a.bound.cpu().numpy())
    assert np.all(a.flag.cpu().numpy() == 0)
