"""GPU GEMM with its row check fused into the kernel, versus the oracle.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method section 2: the checksum and
its check inside the GEMM kernel.  The reference A (W^T 1) is formed by the
kernel's reference warps from the A tiles it stages, against W's column sums
(one pass over W, reusable while W is unchanged).  The product and its row
checksums are the same kernel's as the unfused GEMM's (bit for bit); the
residual, bound and flags are compared with the oracle's.  Since the reference
reads the same staged A tile as the tensor cores, a fault is planted on the
W side: the product reads a corrupted W while the column sums come from the
clean one.
"""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import verifier_own_slack

pytestmark = pytest.mark.gpu
DEV = "cuda"
SHAPES = [(128, 256, 64), (1, 8, 8), (100, 264, 72), (384, 768, 1024), (1000, 2056, 4104), (1024, 2048, 4096)]


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _fused_raise(N: int) -> float:
    """How far above the exact magnitude the fused check's may sit: its plain float32 chains (W's
    column sums, at most N / 8 + 1 rows of one warp; a stage's 32 terms; 8 units of slack) may
    round up by their length and are then raised by twice it, in units of 2^-24."""
    return 3.0 * (N / 8 + 1 + 40) * 2.0 ** -24


def _assert_bound(kb, mb, mag, N, K):
    assert np.all(kb >= mb * (1.0 - 1e-12)), float(np.min(kb / mb))
    top = (mb + verifier_own_slack(N, K) * mag) * (1.0 + _fused_raise(N)) * (1.0 + 1e-12)
    assert np.all(kb <= top), float(np.max(kb / top))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_check_parity(sdc, M, N, K):
    ops = W.gemm_operands(M, N, K, DEV, seed=M + N + K)
    A, Wt = ops["A"], ops["W"]
    g = sdc.AbftGemm(M, N, K, DEV)
    g.weight_sums(Wt)
    g.gemm_checked(A, Wt)
    torch.cuda.synchronize()
    assert int(g.aborted[0]) == 0
    C, rs = g.C.clone(), g.rowsum.clone()
    res, bnd, flag = g.residual.cpu().numpy(), g.bound.cpu().numpy(), g.flag.cpu().numpy()
    # W's column sums: h within its rounding of the exact sums, m an almost exact sum of |W|
    Ab, Wb = _bits(A), _bits(Wt)
    W64 = oracle.bf16_to_f64(Wb)
    ws = g.wsums.cpu().numpy().astype(np.float64)
    absw = np.abs(W64).sum(axis=0)
    assert np.all(np.abs(ws[:, 0] - W64.sum(axis=0)) <= (9.0 * 2.0 ** -24 + (N + 64) * 2.0 ** -44) * absw + 1e-300)
    assert np.all(np.abs(ws[:, 1] - absw) <= (N / 8 + 16) * 2.0 ** -24 * absw + 1e-300)
    # the product and its checksums are the unfused kernel's, bit for bit
    g.gemm(A, Wt)
    torch.cuda.synchronize()
    assert torch.equal(g.C, C) and torch.equal(g.rowsum.view(torch.int64), rs.view(torch.int64))
    # the verdict against the oracle's
    ref, mag = oracle.abft_reference(Ab, Wb)
    v = oracle.abft_verify(rs.cpu().numpy(), Ab, Wb)
    _assert_bound(bnd, v["bound"], mag, N, K)
    assert np.all(np.abs(res - v["residual"]) <= verifier_own_slack(N, K) * mag + 1e-300)
    assert v["n_flagged"] == 0 and np.all(flag == 0) and int(g.summary[0]) == 0 and int(g.summary[1]) == 0


def test_fused_check_agrees_with_the_verifier_and_repeats(sdc):
    M, N, K = 512, 1024, 2048
    ops = W.gemm_operands(M, N, K, DEV, seed=51)
    A, Wt = ops["A"], ops["W"]
    g = sdc.AbftGemm(M, N, K, DEV)
    g.weight_sums(Wt)
    g.gemm_checked(A, Wt)
    r0, b0 = g.residual.clone(), g.bound.clone()
    for _ in range(3):  # the same bits every call, the weight sums reused
        g.gemm_checked(A, Wt)
        assert torch.equal(g.residual.view(torch.int64), r0.view(torch.int64))
        assert torch.equal(g.bound.view(torch.int64), b0.view(torch.int64))
    g.verify(A, Wt)
    torch.cuda.synchronize()
    _, mag = oracle.abft_reference(_bits(A), _bits(Wt))
    # both references are within their own terms of the exact one
    d = np.abs(g.residual.cpu().numpy() - r0.cpu().numpy())
    assert np.all(d <= 2.0 * verifier_own_slack(N, K) * mag)
    assert int(g.summary[0]) == 0


@pytest.mark.parametrize("mask", [0x4000, 0x2000])
def test_fused_check_flags_a_wrong_product(sdc, mask):
    # the product reads W with one element per chosen row of W corrupted, the column sums are the
    # clean W's: every row of C whose exact residual clearly exceeds the bound flags, the others not
    M, N, K = 512, 1024, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=52)
    A, Wt = ops["A"], ops["W"]
    Wf, where = W.gemm_fault(Wt, [3, 500, 777, 1023], seed=53, mask=mask)
    g = sdc.AbftGemm(M, N, K, DEV)
    g.weight_sums(Wt)
    g.gemm_checked(A, Wf)
    torch.cuda.synchronize()
    Ab, Wb, Wfb = _bits(A), _bits(Wt), _bits(Wf)
    with np.errstate(invalid="ignore", over="ignore"):
        exact_rs = oracle.abft_row_checksum(oracle.abft_product(Ab, Wfb))
        v = oracle.abft_verify(exact_rs, Ab, Wb)
    flag = g.flag.cpu().numpy()
    clear = (np.abs(v["residual"]) > 2.0 * v["bound"]) | np.isnan(v["residual"])
    clean = np.abs(v["residual"]) <= 1e-6 * v["bound"]
    assert np.all(flag[clear] == 1) and np.all(flag[clean] == 0)
    assert int(g.summary[0]) == int(flag.sum())
    if mask == 0x4000:
        assert int(clear.sum()) >= M // 2  # a weight 2^128 times larger moves every row


def test_fused_check_rejects_bad_arguments(sdc):
    M, N, K = 128, 256, 64
    ops = W.gemm_operands(M, N, K, DEV, seed=54)
    g = sdc.AbftGemm(M, N, K, DEV)
    with pytest.raises(ValueError):
        g.gemm_checked(ops["A"], ops["W"])  # no weight sums yet
    g.weight_sums(ops["W"])
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm_checked(ops["A"].data_ptr(), ops["W"].data_ptr(), g.C.data_ptr(), M, N, K,
                                  g.wsums.data_ptr(), 0.0, g.rowsum.data_ptr(), g.residual.data_ptr(),
                                  g.bound.data_ptr(), g.flag.data_ptr(), g.summary.data_ptr(), g.aborted.data_ptr(),
                                  g.ws.data_ptr(), g.ws_bytes, 0)
    assert ei.value.status == 9
    assert sdc.sdc_abft_gemm_checked_workspace_size(M, N, K) == 1 * M * 8 + 1 * M * 16 + 256
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_weight_sums(ops["W"].data_ptr(), N, K, g.wsums.data_ptr(), g._wsws.data_ptr(), g._wsb - 256, 0)
    assert ei.value.status == 5
