"""GPU replay context and replay of the GEMM checksum versus the oracle.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method sections 1 and 2: a check
that fires packs the least replay context into a vTask (the forward product:
the flagged row of A and its output row; wgrad: A's rows, B's columns and the
results), which a verifier replays to confirm.

Captures are compared with the oracle's (plain indexing of the same bits),
bit for bit.  A replay of a correct product reproduces every output bit for
bit (the same kernel at the same tile position); a replay of an output that a
fault changed reports every output that the oracle finds inconsistent with
the captured inputs, and more (any bit that differs).
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


def _flags(n: int, picks) -> torch.Tensor:
    f = torch.zeros(n, dtype=torch.uint8, device=DEV)
    f[list(picks)] = 1
    return f


def _check_forward_capture(cap, ref, k_rows: int, k_cols: int):
    n = min(ref["n_rows"], k_rows)
    assert int(cap["counts"][0]) == ref["n_rows"]
    assert cap["row_idx"][:n].cpu().numpy().astype(np.uint32).tolist() == ref["row_idx"].tolist()
    assert np.array_equal(_bits(cap["row_A"][:n]), ref["row_A"])
    assert np.array_equal(_bits(cap["row_C"][:n]), ref["row_C"])
    if "n_cols" in ref:
        m = min(ref["n_cols"], k_cols)
        assert int(cap["counts"][1]) == ref["n_cols"]
        assert cap["col_idx"][:m].cpu().numpy().astype(np.uint32).tolist() == ref["col_idx"].tolist()
        assert np.array_equal(_bits(cap["col_W"][:m]), ref["col_W"])
        assert np.array_equal(_bits(cap["col_C"][:m]), ref["col_C"])


def test_forward_clean_rows_replay_bit_for_bit(sdc):
    # rows at every kind of tile position (first and last lane, either side of a tile edge, the
    # ragged last tile), captured by a chosen selection from a correct product: reproduced exactly
    M, N, K = 1000, 776, 1000
    ops = W.gemm_operands(M, N, K, DEV, seed=41)
    A, Wt = ops["A"], ops["W"]
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g(A, Wt)
    rows, cols = [0, 5, 127, 128, 300, 895, 896, 999], [0, 7, 255, 256, 700, 775]
    cap = g.capture(A, Wt, cap_rows=8, cap_cols=8, flag=_flags(M, rows), flag_col=_flags(N, cols))
    ndiff, summ = g.replay(Wt, cap)
    torch.cuda.synchronize()
    ref = oracle.abft_capture(np.isin(np.arange(M), rows), np.isin(np.arange(N), cols), _bits(A), _bits(Wt),
                              _bits(g.C), 8, 8)
    _check_forward_capture(cap, ref, 8, 8)
    assert ndiff.cpu().tolist() == [0] * 8 and summ.cpu().tolist() == [0, 0]
    assert np.all(oracle.abft_replay_rows(ref["row_A"], _bits(Wt), ref["row_C"]) == 0)


def test_forward_fault_capture_and_replay_confirm(sdc):
    # the GEMM reads a corrupted A, the check the clean one: the flagged rows' context is the clean
    # A row and the computed (wrong) output row; the replay does not reproduce them
    M, N, K = 512, 1024, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=42)
    A, Wt = ops["A"], ops["W"]
    Af, where = W.gemm_fault(A, [3, 100, 257, 384, 511], seed=43, mask=0x4000)
    g = sdc.AbftGemm(M, N, K, DEV)
    g.gemm(Af, Wt)
    g.verify(A, Wt)
    cap = g.capture(A, Wt, cap_rows=4)
    ndiff, summ = g.replay(Wt, cap)
    torch.cuda.synchronize()
    flag = g.flag.cpu().numpy()
    ref = oracle.abft_capture(flag, None, _bits(A), _bits(Wt), _bits(g.C), 4, 0)
    _check_forward_capture(cap, ref, 4, 0)
    assert int(cap["counts"][1]) == 0
    n = min(ref["n_rows"], 4)
    assert n >= 3
    bad = oracle.abft_replay_rows(ref["row_A"], _bits(Wt), ref["row_C"])  # outputs a correct product cannot give
    nd = ndiff.cpu().numpy()[:n]
    assert np.all(bad > 0) and np.all(nd >= bad)
    assert int(summ[0]) == n and int(summ[1]) == 0
    assert np.all(ndiff.cpu().numpy()[n:] == 0)


def test_forward_capture_counts_past_the_cap(sdc):
    M, N, K = 300, 256, 64
    ops = W.gemm_operands(M, N, K, DEV, seed=44)
    g = sdc.AbftGemm(M, N, K, DEV)
    g(ops["A"], ops["W"])
    every = torch.ones(M, dtype=torch.uint8, device=DEV)
    cap = g.capture(ops["A"], ops["W"], cap_rows=4, flag=every)
    ndiff, summ = g.replay(ops["W"], cap)
    torch.cuda.synchronize()
    assert int(cap["counts"][0]) == M and cap["row_idx"].cpu().tolist() == [0, 1, 2, 3]
    assert ndiff.cpu().tolist() == [0, 0, 0, 0] and int(summ[0]) == 0
    none = torch.zeros(M, dtype=torch.uint8, device=DEV)
    cap = g.capture(ops["A"], ops["W"], cap_rows=4, flag=none)
    ndiff, summ = g.replay(ops["W"], cap)
    torch.cuda.synchronize()
    assert int(cap["counts"][0]) == 0 and ndiff.cpu().tolist() == [0] * 4 and int(summ[0]) == 0


def test_wgrad_clean_pairs_replay_bit_for_bit(sdc):
    T, N, K = 1000, 264, 520
    ops = W.wgrad_operands(T, N, K, DEV, seed=45)
    dY, X = ops["dY"], ops["X"]
    a = sdc.AbftWgrad(T, N, K, DEV)
    a(dY, X)
    rows, cols = [0, 127, 128, 263], [0, 255, 256, 519]
    cap = a.capture(dY, X, cap_rows=4, cap_cols=4, flag=_flags(N, rows), flag_col=_flags(K, cols))
    differs, summ = a.replay(cap)
    torch.cuda.synchronize()
    ref = oracle.wgrad_capture(np.isin(np.arange(N), rows), np.isin(np.arange(K), cols), _bits(dY), _bits(X),
                               _bits(a.dW), 4, 4)
    assert cap["counts"].cpu().tolist() == [4, 4]
    for key in ("row_dY", "row_dW", "col_X", "col_dW"):
        assert np.array_equal(_bits(cap[key]), ref[key]), key
    assert differs.cpu().numpy().tolist() == [[0] * 4] * 4 and summ.cpu().tolist() == [0, 0]
    assert np.all(oracle.wgrad_replay_pairs(ref) == 0)


def test_wgrad_fault_capture_and_replay_confirm(sdc):
    # one dY element corrupted for the GEMM: its dW row is flagged, and so are the columns it
    # moved; every (row, column) pair of the captured context fails to reproduce where the oracle
    # finds the saved output inconsistent with the captured operands
    T, N, K = 1024, 512, 768
    ops = W.wgrad_operands(T, N, K, DEV, seed=46)
    dY, X = ops["dY"], ops["X"]
    bad, where = W.gemm_fault(dY, [200], seed=47, mask=0x4000)
    a = sdc.AbftWgrad(T, N, K, DEV)
    a.gemm(bad, X)
    a.verify(dY, X)
    cap = a.capture(dY, X, cap_rows=2, cap_cols=8)
    differs, summ = a.replay(cap)
    torch.cuda.synchronize()
    ref = oracle.wgrad_capture(a.flag.cpu().numpy(), a.flag_col.cpu().numpy(), _bits(dY), _bits(X), _bits(a.dW), 2, 8)
    assert cap["counts"].cpu().tolist() == [ref["n_rows"], ref["n_cols"]]
    assert ref["n_rows"] == 1 and int(ref["row_idx"][0]) == where[0][1] and ref["n_cols"] >= 8
    for key in ("row_dY", "row_dW", "col_X", "col_dW"):
        assert np.array_equal(_bits(cap[key][:len(ref["row_idx"] if key.startswith("row") else ref["col_idx"])]),
                              ref[key]), key
    want = oracle.wgrad_replay_pairs(ref)  # [1, 8]
    got = differs.cpu().numpy()
    assert np.all(got[:1][want == 1] == 1) and want.sum() >= 4
    assert np.all(got[1:] == 0)  # past the captured rows
    assert int(summ[0]) == int(got.sum()) and int(summ[1]) == 0


def test_forward_clean_pairs_replay_bit_for_bit(sdc):
    # the row + column configuration: (row, column) outputs of a correct product, at the tile edges and
    # in the ragged last tiles, recomputed from the captured A rows and W rows alone
    M, N, K = 1000, 776, 1000
    ops = W.gemm_operands(M, N, K, DEV, seed=48)
    A, Wt = ops["A"], ops["W"]
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g(A, Wt)
    rows, cols = [0, 127, 128, 999], [0, 255, 256, 775]
    cap = g.capture(A, Wt, cap_rows=4, cap_cols=4, flag=_flags(M, rows), flag_col=_flags(N, cols))
    differs, summ = g.replay_pairs(cap)
    torch.cuda.synchronize()
    ref = oracle.abft_capture(np.isin(np.arange(M), rows), np.isin(np.arange(N), cols), _bits(A), _bits(Wt),
                              _bits(g.C), 4, 4)
    assert differs.cpu().numpy().tolist() == [[0] * 4] * 4 and summ.cpu().tolist() == [0, 0]
    assert np.all(oracle.abft_replay_pairs(ref) == 0)


def test_forward_fault_pairs_replay_confirm(sdc):
    # the product reads a W with one element of two chosen rows corrupted, the check the clean W: the
    # corrupted rows of W are flagged columns of C; every captured (row, column) pair whose saved
    # output the oracle finds inconsistent with the captured clean operands fails to reproduce
    M, N, K = 512, 1024, 1024
    ops = W.gemm_operands(M, N, K, DEV, seed=49)
    A, Wt = ops["A"], ops["W"]
    Wf, where = W.gemm_fault(Wt, [100, 700], seed=50, mask=0x4000)
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g.gemm(A, Wf)
    g.verify(A, Wt)
    cap = g.capture(A, Wt, cap_rows=4, cap_cols=2)
    differs, summ = g.replay_pairs(cap)
    torch.cuda.synchronize()
    ref = oracle.abft_capture(g.flag.cpu().numpy(), g.flag_col.cpu().numpy(), _bits(A), _bits(Wt), _bits(g.C), 4, 2)
    assert ref["n_cols"] >= 1 and set(ref["col_idx"].tolist()) <= {100, 700}
    want = oracle.abft_replay_pairs(ref)
    got = differs.cpu().numpy()[:len(ref["row_idx"]), :len(ref["col_idx"])]
    assert np.all(got[want == 1] == 1) and want.sum() >= 1
    assert int(summ[0]) == int(differs.sum()) and int(summ[1]) == 0
