"""GPU GEMM with the in-kernel row checksum versus the oracle.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method section 2.  The product C and
the row checksums come from the tensor cores' float32 accumulator, whose
summation order is the hardware's, so they are compared with the oracle's
exact product within the rounding bound; the check's bound, residual and
flags are compared with the oracle's on the kernel's checksums.
"""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import assert_verifier_bound, verifier_own_slack

pytestmark = pytest.mark.gpu
DEV = "cuda"
# one tile; K-blocks past the 4-stage ring (phase wrap); several tiles each way; a larger case
SHAPES = [(128, 256, 64), (256, 512, 320), (384, 768, 1024), (1024, 2048, 4096)]


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _elem_error_bound(Ab, Wb, K):
    """Per-element bound on |float32 accumulator - exact| (the row bound's first and third terms)."""
    mag = np.abs(oracle.bf16_to_f64(Ab)) @ np.abs(oracle.bf16_to_f64(Wb)).T
    g = K * 2.0 ** -22
    return g * (1.0 + g) * mag + 2.0 * K * 2.0 ** -126


def _check_clean(g, Ab, Wb, M, N, K):
    exact = oracle.abft_product(Ab, Wb)
    e = _elem_error_bound(Ab, Wb, K)
    C = g.C.float().cpu().numpy().astype(np.float64)
    # round-to-nearest into bf16 moves a value by at most 2^-8 of itself (2^-134 if subnormal)
    tol = 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134
    assert np.all(np.abs(C - exact) <= tol), np.max(np.abs(C - exact) / tol)
    rs = g.rowsum.cpu().numpy()
    _, mag = oracle.abft_reference(Ab, Wb)
    bound = oracle.abft_bound(mag, N, K)
    assert np.all(np.abs(rs - oracle.abft_row_checksum(exact)) <= bound)
    v = oracle.abft_verify(rs, Ab, Wb, tol_scale=1.0)
    # the kernel's bound adds its own terms to the method's (float32-pair sums, a raised plain
    # float32 magnitude); its reference sums agree with the oracle's float64 to the pair term
    eps = verifier_own_slack(N, K)
    assert_verifier_bound(g.bound.cpu().numpy(), v["bound"], mag, N, K)
    res = g.residual.cpu().numpy()
    assert np.all(np.abs(res - v["residual"]) <= eps * mag)
    assert np.all(g.flag.cpu().numpy() == 0) and v["n_flagged"] == 0
    assert int(g.summary[0]) == 0
    assert int(g.aborted[0]) == 0
    return float(np.max(np.abs(res) / v["bound"]))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_checksum_parity(sdc, M, N, K):
    ops = W.gemm_operands(M, N, K, DEV, seed=M + N + K)
    g = sdc.AbftGemm(M, N, K, DEV)
    g(ops["A"], ops["W"])
    torch.cuda.synchronize()
    ratio = _check_clean(g, _bits(ops["A"]), _bits(ops["W"]), M, N, K)
    assert ratio < 0.5  # the float32 rounding noise is far inside the bound


def test_matches_torch_matmul(sdc):
    # the same product from cuBLAS: both round a float32 accumulation to bf16, in
    # different orders, so they agree within two bf16 units of the accumulator bound
    M, N, K = 512, 1024, 2048
    ops = W.gemm_operands(M, N, K, DEV, seed=21)
    g = sdc.AbftGemm(M, N, K, DEV)
    C = g(ops["A"], ops["W"]).float().cpu().numpy().astype(np.float64)
    ref = (ops["A"] @ ops["W"].t()).float().cpu().numpy().astype(np.float64)
    e = _elem_error_bound(_bits(ops["A"]), _bits(ops["W"]), K)
    assert np.all(np.abs(C - ref) <= 2.0 ** -7 * (np.abs(ref) + 2 * e) + 2 * e + 2.0 ** -133)


def test_deterministic_and_reusable(sdc):
    M, N, K = 256, 512, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=22)
    g = sdc.AbftGemm(M, N, K, DEV)
    g(ops["A"], ops["W"])
    C0, rs0 = g.C.clone(), g.rowsum.clone()
    for _ in range(3):
        g(ops["A"], ops["W"])
        assert torch.equal(g.C, C0)
        assert torch.equal(g.rowsum.view(torch.int64), rs0.view(torch.int64))
    # a second shape on the same stream
    ops2 = W.gemm_operands(128, 256, 128, DEV, seed=23)
    g2 = sdc.AbftGemm(128, 256, 128, DEV)
    g2(ops2["A"], ops2["W"])
    torch.cuda.synchronize()
    _check_clean(g2, _bits(ops2["A"]), _bits(ops2["W"]), 128, 256, 128)


@pytest.mark.parametrize("mask", [0x4000, 0x2000, 0x0080])
def test_operand_fault_flags_its_rows(sdc, mask):
    # the GEMM reads a corrupted A (one element of each planted row XORed with `mask`),
    # the check uses the clean A: rows whose exact residual is clearly above the bound
    # flag, rows with no fault do not
    M, N, K = 512, 1024, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=24)
    A, Wt = ops["A"], ops["W"]
    rows = [0, 3, 100, 257, 384, 511]
    Af, where = W.gemm_fault(A, rows, seed=mask, mask=mask)
    g = sdc.AbftGemm(M, N, K, DEV)
    g.gemm(Af, Wt)
    g.verify(A, Wt, tol_scale=1.0)
    torch.cuda.synchronize()
    Ab, Afb, Wb = _bits(A), _bits(Af), _bits(Wt)
    with np.errstate(invalid="ignore", over="ignore"):
        exact_rs = oracle.abft_row_checksum(oracle.abft_product(Afb, Wb))
    v = oracle.abft_verify(exact_rs, Ab, Wb, tol_scale=1.0)
    flag = g.flag.cpu().numpy()
    clear = (np.abs(v["residual"]) > 2.0 * v["bound"]) | np.isnan(v["residual"])
    # untouched outputs: the oracle's two float64 sums differ only by their own rounding
    clean = np.abs(v["residual"]) <= 1e-6 * v["bound"]
    assert np.all(flag[clear] == 1)
    assert np.all(flag[clean] == 0)
    assert set(np.nonzero(~clean)[0]) <= set(rows)
    assert int(g.summary[0]) == int(flag.sum())
    if mask == 0x4000:  # the top exponent bit: NaN, infinities or values near 2^128
        assert int(clear.sum()) >= 4


def test_rejects_misaligned_and_short_workspace(sdc):
    M, N, K = 128, 256, 64
    ops = W.gemm_operands(M, N, K + 8, DEV, seed=25)
    g = sdc.AbftGemm(M, N, K, DEV)
    A_odd = ops["A"].view(-1)[1:1 + M * K]  # 2-byte offset
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm(A_odd.data_ptr(), ops["W"].data_ptr(), g.C.data_ptr(), M, N, K, g.rowsum.data_ptr(), 0,
                          g.aborted.data_ptr(), g.ws.data_ptr(), g.ws_bytes, 0)
    assert ei.value.status == 8
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm(ops["A"].data_ptr(), ops["W"].data_ptr(), g.C.data_ptr(), M, N, K, g.rowsum.data_ptr(), 0,
                          g.aborted.data_ptr(), g.ws.data_ptr(), g.ws_bytes - 256, 0)
    assert ei.value.status == 5


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_row_and_column_checksums(sdc, M, N, K):
    # the page's row + column configuration: 1^T C from the accumulator against (1^T A) W^T
    ops = W.gemm_operands(M, N, K, DEV, seed=M + N + K)
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g(ops["A"], ops["W"])
    r = sdc.AbftGemm(M, N, K, DEV)
    r(ops["A"], ops["W"])
    torch.cuda.synchronize()
    Ab, Wb = _bits(ops["A"]), _bits(ops["W"])
    _check_clean(g, Ab, Wb, M, N, K)
    # the row side and the product do not change with the column side on
    assert torch.equal(g.C, r.C) and torch.equal(g.rowsum.view(torch.int64), r.rowsum.view(torch.int64))
    exact = oracle.abft_product(Ab, Wb)
    cs = g.colsum.cpu().numpy()
    v = oracle.abft_verify_cols(cs, Ab, Wb)
    assert np.all(np.abs(cs - exact.sum(axis=0)) <= v["bound"])
    eps = verifier_own_slack(M, K)
    _, mag = oracle.abft_reference_cols(Ab, Wb)
    assert_verifier_bound(g.bound_col.cpu().numpy(), v["bound"], mag, M, K)
    assert np.all(np.abs(g.residual_col.cpu().numpy() - v["residual"]) <= eps * mag)
    assert np.all(g.flag_col.cpu().numpy() == 0) and int(g.summary[1]) == 0
    assert float(np.max(np.abs(v["residual"]) / v["bound"])) < 0.5


def test_weight_fault_flags_its_columns(sdc):
    # the GEMM reads a corrupted W (one element of each planted row of W, i.e. output column,
    # XORed with the top exponent bit), the check uses the clean W
    M, N, K = 512, 1024, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=26)
    A, Wt = ops["A"], ops["W"]
    cols = [0, 17, 300, 1023]
    Wf, where = W.gemm_fault(Wt, cols, seed=27, mask=0x4000)
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g.gemm(A, Wf)
    g.verify(A, Wt)
    torch.cuda.synchronize()
    Ab, Wb, Wfb = _bits(A), _bits(Wt), _bits(Wf)
    with np.errstate(invalid="ignore", over="ignore"):
        exact_cs = oracle.abft_product(Ab, Wfb).sum(axis=0)
    v = oracle.abft_verify_cols(exact_cs, Ab, Wb)
    flag = g.flag_col.cpu().numpy()
    clear = (np.abs(v["residual"]) > 2.0 * v["bound"]) | np.isnan(v["residual"])
    # untouched outputs: the oracle's two float64 sums differ only by their own rounding
    clean = np.abs(v["residual"]) <= 1e-6 * v["bound"]
    assert np.all(flag[clear] == 1) and np.all(flag[clean] == 0)
    assert set(np.nonzero(~clean)[0]) <= set(cols)
    assert int(clear.sum()) >= 2
    assert int(g.summary[1]) == int(flag.sum())


def test_largest_contraction(sdc):
    # the largest K the kernel accepts (2^20), where the rounding bound is at its loosest
    # (g = K 2^-22 = 1/4): one tile, rows and columns, against the oracle
    M, N, K = 128, 256, 1 << 20
    ops = W.gemm_operands(M, N, K, DEV, seed=41)
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g(ops["A"], ops["W"])
    torch.cuda.synchronize()
    Ab, Wb = _bits(ops["A"]), _bits(ops["W"])
    del ops
    _check_clean(g, Ab, Wb, M, N, K)
    cs = g.colsum.cpu().numpy()
    v = oracle.abft_verify_cols(cs, Ab, Wb)
    assert v["n_flagged"] == 0 and int(g.summary[1]) == 0 and np.all(g.flag_col.cpu().numpy() == 0)


RAGGED = [(1, 8, 8), (100, 264, 72), (129, 520, 1000), (200, 776, 4104), (300, 256, 64)]


@pytest.mark.parametrize("columns", [False, True])
@pytest.mark.parametrize("M,N,K", RAGGED)
def test_ragged_shapes(sdc, M, N, K, columns):
    # shapes that are not multiples of the 128 x 256 x 64 tiles (any M, N and K multiples of 8): the
    # copies fill the tiles' rows and columns outside A and W with zeros, the epilogue stores
    # only inside C; odd and even tile-row counts
    ops = W.gemm_operands(M, N, K, DEV, seed=70 + M + N + K)
    g = sdc.AbftGemm(M, N, K, DEV, columns=columns)
    g(ops["A"], ops["W"])
    torch.cuda.synchronize()
    Ab, Wb = _bits(ops["A"]), _bits(ops["W"])
    _check_clean(g, Ab, Wb, M, N, K)
    if columns:
        exact = oracle.abft_product(Ab, Wb)
        cs = g.colsum.cpu().numpy()
        v = oracle.abft_verify_cols(cs, Ab, Wb)
        assert np.all(np.abs(cs - exact.sum(axis=0)) <= v["bound"])
        assert v["n_flagged"] == 0 and int(g.summary[1]) == 0 and np.all(g.flag_col.cpu().numpy() == 0)


@pytest.mark.parametrize("M,N,K", [(100, 264, 72), (129, 520, 1000)])
def test_ragged_stores_stay_inside_c(sdc, M, N, K):
    # through the C ABI with C followed by a sentinel region: nothing past M x N is written
    ops = W.gemm_operands(M, N, K, DEV, seed=80 + M)
    buf = torch.full((M * N + 8192,), 0x7777, dtype=torch.int16, device=DEV)
    rowsum = torch.empty(M, dtype=torch.float64, device=DEV)
    colsum = torch.empty(N, dtype=torch.float64, device=DEV)
    aborted = torch.zeros(1, dtype=torch.int32, device=DEV)
    nws = sdc.sdc_abft_workspace_size(M, N, K)
    ws = torch.empty(nws + 256, dtype=torch.uint8, device=DEV)
    wsp = (ws.data_ptr() + 255) // 256 * 256
    sdc.sdc_abft_gemm(ops["A"].data_ptr(), ops["W"].data_ptr(), buf.data_ptr(), M, N, K, rowsum.data_ptr(),
                      colsum.data_ptr(), aborted.data_ptr(), wsp, nws, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(aborted[0]) == 0
    assert bool((buf[M * N:] == 0x7777).all())
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g.gemm(ops["A"], ops["W"])
    torch.cuda.synchronize()
    assert torch.equal(buf[:M * N].view(M, N), g.C.view(torch.int16))
    assert torch.equal(rowsum.view(torch.int64), g.rowsum.view(torch.int64))
    assert torch.equal(colsum.view(torch.int64), g.colsum.view(torch.int64))
