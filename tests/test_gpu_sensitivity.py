"""How small a planted fault the two tensor-core checks catch at tol_scale 1.

[AEGIS] method sections 2 and 3 give no thresholds, so these sweeps measure
the smallest fault that flags, against the oracle:
- the GEMM row checksum: one A element per row with one bit flipped, for
  every bit of the bf16 pattern;
- the attention invariant: one row's log-sum-exp shifted by -2^k or +2^k,
  and one K element with one bit flipped.
In every case a row or column whose exact residual (the oracle's, from the
faulty inputs) is beyond twice the bound must flag, and one inside a tenth of
it must not.  The thresholds found are printed (run with -s to see them).
"""
import json

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


def test_gemm_bit_sweep(sdc):
    M, N, K = 256, 1024, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=91)
    A, Wt = ops["A"], ops["W"]
    Ab, Wb = _bits(A), _bits(Wt)
    A64, W64 = oracle.bf16_to_f64(Ab), oracle.bf16_to_f64(Wb)
    colW = W64.sum(axis=0)
    ref, mag = oracle.abft_reference(Ab, Wb)
    bound = oracle.abft_bound(mag, N, K)
    rng = np.random.default_rng(92)
    rows = np.sort(rng.choice(M, 32, replace=False))
    g = sdc.AbftGemm(M, N, K, DEV)
    summary = {}
    for bit in range(15):  # the sign bit is bit 15; 0-6 mantissa, 7-14 exponent
        Af, where = W.gemm_fault(A, [int(r) for r in rows], seed=100 + bit, mask=1 << bit)
        g.gemm(Af, Wt)
        g.verify(A, Wt, tol_scale=1.0)
        torch.cuda.synchronize()
        flag = g.flag.cpu().numpy()
        Afb = _bits(Af)
        with np.errstate(over="ignore", invalid="ignore"):
            delta = oracle.bf16_to_f64(Afb[rows]) - A64[rows]  # one non-zero per planted row
            r = (delta * colW[None, :]).sum(axis=1)  # exact change of the row checksum
        ratio = np.abs(r) / bound[rows]
        clear = (ratio > 2.0) | np.isnan(r)
        clean = ratio < 0.1
        assert np.all(flag[rows][clear] == 1), (bit, ratio[clear & (flag[rows] == 0)])
        assert np.all(flag[rows][clean] == 0), (bit, ratio[clean & (flag[rows] == 1)])
        others = np.setdiff1d(np.arange(M), rows)
        assert np.all(flag[others] == 0)  # untouched rows never flag
        fl = flag[rows] == 1
        summary[bit] = {"flagged": int(fl.sum()), "of": len(rows),
                        "smallest_flagged_ratio": float(ratio[fl].min()) if fl.any() else None,
                        "largest_unflagged_ratio": float(ratio[~fl].max()) if (~fl).any() else None}
        if bit == 14:  # the top exponent bit: a value it makes 2^128 times larger (or Inf/NaN) always flags
            with np.errstate(over="ignore", invalid="ignore"):
                grown = ~(np.abs(delta).max(axis=1) < 1e30)
            assert grown.any() and np.all(fl[grown])
    print("\nGEMM row checksum, 256 x 1024 x 1024, one A bit per row:", json.dumps(summary))


def _attn_expected(x, Kb_used, lse_used, h):
    Qb, dOb = _bits(x["Q"]), _bits(x["dO"])
    with np.errstate(over="ignore", invalid="ignore"):
        P = oracle.attn_probs(Qb[h], Kb_used[h], lse_used[h], x["scale"], x["causal"])
        v = oracle.attn_invariant(oracle.attn_dv(P, dOb[h]).sum(axis=0), dOb[h])
    return np.abs(v["residual"]) / v["bound"], v["residual"]


def _max_ratio(ratio) -> float:
    """The largest residual / bound, a NaN residual counting as infinitely beyond the bound."""
    return float(np.max(np.where(np.isnan(ratio), np.inf, ratio)))


def _attn_run(sdc, x):
    BH, L, _ = x["Q"].shape
    a = sdc.AttnDvCheck(BH, L, DEV)
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], x["causal"], 1.0)
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0
    return a


def test_attention_lse_shift_sweep(sdc):
    x = W.attn_inputs(1, 512, DEV, seed=93, causal=False)
    summary = {}
    for k in range(-8, 3):
        for sign in (-1.0, 1.0):
            d = sign * 2.0 ** k
            bad = x["lse"].clone()
            bad[0, 200] += d
            a = _attn_run(sdc, dict(x, lse=bad))
            ratio, res = _attn_expected(x, _bits(x["K"]), bad.cpu().numpy(), 0)
            flag = a.flag[0].cpu().numpy()
            assert np.all(flag[(ratio > 2.0) | np.isnan(res)] == 1), d
            assert np.all(flag[ratio < 0.1] == 0), d
            summary[d] = {"columns_flagged": int(flag.sum()), "of": 128, "max_ratio": _max_ratio(ratio)}
    # a shift of -4 multiplies the row by e^4: most columns clear the bound
    assert summary[-4.0]["columns_flagged"] >= 64
    print("\nattention invariant, 1 x 512 x 128, one row's log-sum-exp shifted by d:", json.dumps(summary))


def test_attention_key_bit_sweep(sdc):
    x = W.attn_inputs(1, 512, DEV, seed=94, causal=False)
    summary = {}
    for bit in range(15):
        Kf = x["K"].clone()
        W.xor_element(Kf, 300 * 128 + 40, 1 << bit)
        a = _attn_run(sdc, dict(x, K=Kf))
        ratio, res = _attn_expected(x, _bits(Kf), x["lse"].cpu().numpy(), 0)
        flag = a.flag[0].cpu().numpy()
        assert np.all(flag[(ratio > 2.0) | np.isnan(res)] == 1), bit
        assert np.all(flag[ratio < 0.1] == 0), bit
        summary[bit] = {"columns_flagged": int(flag.sum()), "of": 128, "max_ratio": _max_ratio(ratio)}
    print("\nattention invariant, 1 x 512 x 128, one K element's bit flipped:", json.dumps(summary))
