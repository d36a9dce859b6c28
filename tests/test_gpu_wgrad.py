"""GPU weight-gradient GEMM with row and column checksums versus the oracle.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method section 2: the row + column
configuration of the accumulator checksum covers every matmul class, the
weight gradient (wgrad) included.  dW = dY^T X with dY [T, N] and X [T, K]
token-major; the operands reach the tensor cores MN-major.  dW and both
checksums come from the float32 accumulator in the hardware's order, so they
are compared with the oracle's exact values within the rounding bound; the
check's bounds, residuals and flags with the oracle's on the kernel's
checksums.
"""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import assert_wgrad_bound, verifier_own_slack

pytestmark = pytest.mark.gpu
DEV = "cuda"
# one tile; ragged T, N and K; contraction past the 4-stage ring; one token; the smallest shape;
# several tiles each way with a long contraction
SHAPES = [(64, 128, 256), (1000, 264, 520), (320, 384, 768), (1, 128, 256), (8, 8, 8), (4096, 1024, 2048)]


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_clean(a, dYb, Xb, T, N, K):
    exact = oracle.wgrad_product(dYb, Xb)
    g = T * 2.0 ** -22
    e = g * (1.0 + g) * (np.abs(oracle.bf16_to_f64(dYb)).T @ np.abs(oracle.bf16_to_f64(Xb))) + 2.0 * T * 2.0 ** -126
    dW = a.dW.float().cpu().numpy().astype(np.float64)
    # round-to-nearest into bf16 moves a value by at most 2^-8 of itself (2^-134 if subnormal)
    tol = 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134
    assert np.all(np.abs(dW - exact) <= tol), np.max(np.abs(dW - exact) / tol)
    ref = oracle.wgrad_reference(dYb, Xb)
    rs, cs = a.rowsum.cpu().numpy(), a.colsum.cpu().numpy()
    assert np.all(np.abs(rs - exact.sum(axis=1)) <= oracle.abft_bound(ref["row_mag"], K, T))
    assert np.all(np.abs(cs - exact.sum(axis=0)) <= oracle.abft_bound(ref["col_mag"], N, T))
    v = oracle.wgrad_verify(rs, cs, dYb, Xb)
    assert_wgrad_bound(a.bound.cpu().numpy(), v["bound"], ref["row_mag"], K, T)
    assert_wgrad_bound(a.bound_col.cpu().numpy(), v["bound_col"], ref["col_mag"], N, T)
    # the kernel's references agree with the oracle's float64 ones to its own term
    assert np.all(np.abs(a.residual.cpu().numpy() - v["residual"]) <= verifier_own_slack(K, T) * ref["row_mag"])
    assert np.all(np.abs(a.residual_col.cpu().numpy() - v["residual_col"]) <= verifier_own_slack(N, T) * ref["col_mag"])
    assert v["n_flagged"] == 0 and v["n_flagged_col"] == 0
    assert np.all(a.flag.cpu().numpy() == 0) and np.all(a.flag_col.cpu().numpy() == 0)
    assert int(a.summary[0]) == 0 and int(a.summary[1]) == 0 and int(a.aborted[0]) == 0


@pytest.mark.parametrize("T,N,K", SHAPES)
def test_wgrad_checksum_parity(sdc, T, N, K):
    ops = W.wgrad_operands(T, N, K, DEV, seed=T + N + K)
    a = sdc.AbftWgrad(T, N, K, DEV)
    a(ops["dY"], ops["X"])
    torch.cuda.synchronize()
    _check_clean(a, _bits(ops["dY"]), _bits(ops["X"]), T, N, K)


def test_matches_torch_matmul(sdc):
    # cuBLAS's dY^T X rounds another float32 accumulation order to bf16: within two bf16 units
    T, N, K = 2048, 512, 1024
    ops = W.wgrad_operands(T, N, K, DEV, seed=31)
    a = sdc.AbftWgrad(T, N, K, DEV)
    dW = a(ops["dY"], ops["X"]).float().cpu().numpy().astype(np.float64)
    ref = (ops["dY"].t() @ ops["X"]).float().cpu().numpy().astype(np.float64)
    g = T * 2.0 ** -22
    e = g * (1 + g) * (np.abs(oracle.bf16_to_f64(_bits(ops["dY"]))).T @ np.abs(oracle.bf16_to_f64(_bits(ops["X"]))))
    e += 2.0 * T * 2.0 ** -126
    assert np.all(np.abs(dW - ref) <= 2.0 ** -7 * (np.abs(ref) + 2 * e) + 2 * e + 2.0 ** -133)


def test_deterministic_reusable_and_rows_only(sdc):
    T, N, K = 640, 256, 512
    ops = W.wgrad_operands(T, N, K, DEV, seed=32)
    a = sdc.AbftWgrad(T, N, K, DEV)
    a(ops["dY"], ops["X"])
    dW0, rs0, cs0, b0 = a.dW.clone(), a.rowsum.clone(), a.colsum.clone(), a.bound_col.clone()
    for _ in range(3):
        a(ops["dY"], ops["X"])
        assert torch.equal(a.dW, dW0)
        assert torch.equal(a.rowsum.view(torch.int64), rs0.view(torch.int64))
        assert torch.equal(a.colsum.view(torch.int64), cs0.view(torch.int64))
        assert torch.equal(a.bound_col.view(torch.int64), b0.view(torch.int64))
    # rows only: the same dW and row checksums, the row check alone
    r = sdc.AbftWgrad(T, N, K, DEV, columns=False)
    r(ops["dY"], ops["X"])
    torch.cuda.synchronize()
    assert torch.equal(r.dW, dW0) and torch.equal(r.rowsum.view(torch.int64), rs0.view(torch.int64))
    assert torch.equal(r.bound, a.bound) and int(r.summary[0]) == 0 and int(r.summary[1]) == 0


@pytest.mark.parametrize("operand", ["dY", "X"])
def test_operand_fault_flags_rows_and_columns(sdc, operand):
    # the GEMM reads a corrupted operand (one element of each listed token's row XORed with the
    # top exponent bit), the check the clean one: outputs whose exact residual is clearly above
    # the bound flag, untouched ones do not
    T, N, K = 1024, 512, 768
    ops = W.wgrad_operands(T, N, K, DEV, seed=33)
    dY, X = ops["dY"], ops["X"]
    tokens = [0, 17, 500, 1023]
    bad, where = W.gemm_fault(dY if operand == "dY" else X, tokens, seed=34, mask=0x4000)
    a = sdc.AbftWgrad(T, N, K, DEV)
    if operand == "dY":
        a.gemm(bad, X)
    else:
        a.gemm(dY, bad)
    a.verify(dY, X, tol_scale=1.0)
    torch.cuda.synchronize()
    dYb, Xb, badb = _bits(dY), _bits(X), _bits(bad)
    with np.errstate(invalid="ignore", over="ignore"):
        exact = oracle.wgrad_product(badb, Xb) if operand == "dY" else oracle.wgrad_product(dYb, badb)
        v = oracle.wgrad_verify(exact.sum(axis=1), exact.sum(axis=0), dYb, Xb)
    clears = {}
    for tag, flag in (("", a.flag), ("_col", a.flag_col)):
        f = flag.cpu().numpy()
        res, bnd = v["residual" + tag], v["bound" + tag]
        clear = (np.abs(res) > 2.0 * bnd) | np.isnan(res)
        clean = np.abs(res) <= 1e-6 * bnd
        assert np.all(f[clear] == 1), tag
        assert np.all(f[clean] == 0), tag
        clears[tag] = set(np.nonzero(clear)[0].tolist())
    # a faulty dY element touches one row of dW (its column n) and every column; a faulty X
    # element one column (its k) and every row: on that side only the hit outputs can flag
    hit = {c for _, c in where}
    tag = "" if operand == "dY" else "_col"
    flagged = set(np.nonzero((a.flag if operand == "dY" else a.flag_col).cpu().numpy())[0].tolist())
    assert clears[tag] <= flagged <= hit and len(clears[tag]) >= 2
    assert int(a.summary[0]) == int(a.flag.sum()) and int(a.summary[1]) == int(a.flag_col.sum())


def test_rejects_misaligned_and_short_workspace(sdc):
    T, N, K = 128, 256, 64
    ops = W.wgrad_operands(T, N, K + 8, DEV, seed=35)
    a = sdc.AbftWgrad(T, N, K, DEV)
    X_odd = ops["X"].view(-1)[1:1 + T * K]  # 2-byte offset
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm_wgrad(ops["dY"].data_ptr(), X_odd.data_ptr(), a.dW.data_ptr(), T, N, K,
                                a.rowsum.data_ptr(), 0, a.aborted.data_ptr(), a.ws.data_ptr(), a.ws_bytes, 0)
    assert ei.value.status == 8
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_verify_wgrad(ops["dY"].data_ptr(), X_odd.data_ptr(), T, N, K, a.rowsum.data_ptr(), 0, 1.0,
                                  a.residual.data_ptr(), a.bound.data_ptr(), a.flag.data_ptr(), 0, 0, 0,
                                  a.summary.data_ptr(), a.ws.data_ptr(), a.ws_bytes - 256, 0)
    assert ei.value.status in (5, 8)
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm_wgrad(ops["dY"].data_ptr(), ops["X"].data_ptr(), a.dW.data_ptr(), T, N, K,
                                a.rowsum.data_ptr(), 0, a.aborted.data_ptr(), a.ws.data_ptr(), a.ws_bytes - 256, 0)
    assert ei.value.status == 5


def test_wgrad_largest_contraction(sdc):
    # the most tokens the kernel accepts (2^20), where the rounding bound is at its loosest
    # (g = T 2^-22 = 1/4): one tile, rows and columns, against the oracle
    T, N, K = 1 << 20, 8, 64
    ops = W.wgrad_operands(T, N, K, DEV, seed=36)
    a = sdc.AbftWgrad(T, N, K, DEV)
    a(ops["dY"], ops["X"])
    torch.cuda.synchronize()
    dYb, Xb = _bits(ops["dY"]), _bits(ops["X"])
    del ops
    _check_clean(a, dYb, Xb, T, N, K)
    with pytest.raises(sdc.SdcError) as ei:  # one token more is rejected
        sdc.AbftWgrad(T + 8, N, K, DEV).gemm(torch.empty((T + 8, N), dtype=torch.bfloat16, device=DEV),
                                             torch.empty((T + 8, K), dtype=torch.bfloat16, device=DEV))
    assert ei.value.status == 9
