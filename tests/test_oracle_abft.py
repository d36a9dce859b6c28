"""Pins of the oracle's GEMM checksum.

Source: "Safeguarding LLM Training at Scale: Online SDC Detection and Insights
from 35 Million GPU Hours" (review page), method section 2: the matrix checksum
compares (AB)1 with A(B1), the checksum taken from the float32 accumulator
before the bfloat16 output is rounded.  Here the product is C = A W^T (a linear
layer's forward pass), so B1 = W^T 1.

Each pin is independent of the oracle's own arithmetic: pure-Python integer and
Fraction brute force, closed forms for planted operand faults, and an emulation
of float32 accumulation (round-to-nearest and truncating, per step and per
16-wide block) against which the rounding bound must hold.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values that are exact in bfloat16 -> their bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0), "value not exact in bf16"
    return (b >> 16).astype(np.uint16)


def _bf16_round(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _int_operands(M, N, K, seed, lo=-16, hi=16):
    rng = np.random.default_rng(seed)
    A = rng.integers(lo, hi + 1, size=(M, K))
    W = rng.integers(lo, hi + 1, size=(N, K))
    return A, W, _bf16_bits(A.astype(np.float32)), _bf16_bits(W.astype(np.float32))


def test_bf16_decode_fixed_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0xFF80, 0x0001, 0x4049], dtype=np.uint16)
    v = oracle.bf16_to_f64(bits)
    assert list(v[:6]) == [1.0, -2.0, 0.0, -0.0, np.inf, -np.inf]
    assert v[6] == 2.0 ** -133  # smallest subnormal
    assert v[7] == 3.140625  # 0x4049: 1.5703125 * 2
    assert np.isnan(oracle.bf16_to_f64(np.array([0x7FC0], dtype=np.uint16))[0])


def test_product_matches_fraction_brute_force():
    # non-square shapes so a transposed operand cannot pass; dyadic values exact in bf16
    M, N, K = 3, 5, 7
    rng = np.random.default_rng(1)
    A = (rng.integers(-255, 256, size=(M, K)) * 2.0 ** rng.integers(-20, 20, size=(M, K))).astype(np.float32)
    W = (rng.integers(-255, 256, size=(N, K)) * 2.0 ** rng.integers(-20, 20, size=(N, K))).astype(np.float32)
    Ab, Wb = _bf16_bits(A), _bf16_bits(W)
    C = oracle.abft_product(Ab, Wb)
    assert C.shape == (M, N)
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(float(A[i, k])) * Fraction(float(W[j, k])) for k in range(K))
            assert abs(Fraction(C[i, j]) - exact) <= Fraction(K) * Fraction(2) ** -52 * sum(
                abs(Fraction(float(A[i, k])) * Fraction(float(W[j, k]))) for k in range(K))


def test_checksum_identity_on_integers():
    # integer data: every sum is exact, so (A W^T) 1 == A (W^T 1) holds with equality
    M, N, K = 16, 24, 40
    A, W, Ab, Wb = _int_operands(M, N, K, 2)
    rowsum = oracle.abft_row_checksum(oracle.abft_product(Ab, Wb))
    ref, mag = oracle.abft_reference(Ab, Wb)
    brute = [sum(int(A[i, k]) * int(W[j, k]) for j in range(N) for k in range(K)) for i in range(M)]
    brute_mag = [sum(abs(int(A[i, k])) * abs(int(W[j, k])) for j in range(N) for k in range(K)) for i in range(M)]
    assert list(rowsum) == brute
    assert list(ref) == brute
    assert list(mag) == brute_mag
    v = oracle.abft_verify(rowsum, Ab, Wb)
    assert v["n_flagged"] == 0 and np.all(v["residual"] == 0)


@pytest.mark.parametrize("delta", [1, -3, 7])
def test_planted_operand_fault_closed_form(delta):
    # the GEMM reads A' = A + delta e_(i,k); the check uses A: the residual of row i
    # is delta * sum_j W[j, k] and every other row's is zero
    M, N, K = 8, 12, 20
    A, W, Ab, Wb = _int_operands(M, N, K, 3, lo=-8, hi=8)
    i, k = 5, 11
    Af = A.copy()
    Af[i, k] += delta
    rowsum = oracle.abft_row_checksum(oracle.abft_product(_bf16_bits(Af.astype(np.float32)), Wb))
    v = oracle.abft_verify(rowsum, Ab, Wb, tol_scale=1.0)
    expect = np.zeros(M)
    expect[i] = delta * int(W[:, k].sum())
    assert np.array_equal(v["residual"], expect)
    # integers: the bound is far below 1, so the row flags exactly when the column sum is non-zero
    assert v["n_flagged"] == int(W[:, k].sum() != 0)
    assert v["flag"][i] == int(W[:, k].sum() != 0)


def _emulate_fp32(Af: np.ndarray, Wf: np.ndarray, mode: str) -> np.ndarray:
    """float32 accumulators of A W^T: per-step round-to-nearest, per-step truncation,
    or 16-wide blocks summed exactly then truncated into the accumulator."""
    M, K = Af.shape
    N = Wf.shape[0]
    acc = np.zeros((M, N), dtype=np.float64)

    def trunc32(x):
        r = x.astype(np.float32).astype(np.float64)
        over = np.abs(r) > np.abs(x)
        r[over] = np.nextafter(r[over].astype(np.float32), np.float32(0)).astype(np.float64)
        return r

    if mode == "block16":
        for k0 in range(0, K, 16):
            blk = acc + Af[:, k0:k0 + 16] @ Wf[:, k0:k0 + 16].T
            acc = trunc32(blk)
        return acc
    for k in range(K):
        x = acc + np.outer(Af[:, k], Wf[:, k])  # the product of two bf16 is exact in float64
        acc = x.astype(np.float32).astype(np.float64) if mode == "rn" else trunc32(x)
    return acc


@pytest.mark.parametrize("mode", ["rn", "trunc", "block16"])
@pytest.mark.parametrize("dist", ["normal", "positive", "dominant", "wide"])
def test_bound_covers_float32_accumulation(mode, dist):
    M, N, K = 8, 32, 512
    rng = np.random.default_rng(4)
    if dist == "normal":
        A32 = rng.standard_normal((M, K)).astype(np.float32)
        W32 = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    elif dist == "positive":  # no cancellation: partial sums grow, rounding errors add up
        A32 = rng.uniform(0.5, 1.0, (M, K)).astype(np.float32)
        W32 = rng.uniform(0.5, 1.0, (N, K)).astype(np.float32)
    elif dist == "dominant":  # positive, over 12 binades, one large first term: every later
        # product is added to a partial sum whose unit in the last place exceeds its low bits
        A32 = (rng.uniform(0.5, 1.0, (M, K)) * 2.0 ** -rng.integers(0, 12, (M, K))).astype(np.float32)
        W32 = (rng.uniform(0.5, 1.0, (N, K)) * 2.0 ** -rng.integers(0, 12, (N, K))).astype(np.float32)
        A32[:, 0], W32[:, 0] = 2.0 ** 10, 2.0 ** 4
    else:  # magnitudes over 40 binades
        A32 = (rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, (M, K))).astype(np.float32)
        W32 = (rng.standard_normal((N, K)) * 2.0 ** rng.integers(-20, 20, (N, K))).astype(np.float32)
    Ab, Wb = _bf16_round(A32), _bf16_round(W32)
    acc = _emulate_fp32(oracle.bf16_to_f64(Ab), oracle.bf16_to_f64(Wb), mode)
    v = oracle.abft_verify(acc.sum(axis=1), Ab, Wb, tol_scale=1.0)
    assert v["n_flagged"] == 0
    ratio = np.max(np.abs(v["residual"]) / v["bound"])
    assert ratio <= 1.0
    # not vacuous: to first order the bound is K 2^-22 of the magnitude
    _, mag = oracle.abft_reference(Ab, Wb)
    assert np.all(v["bound"] <= 1.01 * K * 2.0 ** -22 * mag + 1e-30)
    if dist == "dominant" and mode == "trunc":
        assert ratio > 0.05  # one-sided truncation errors add up to a sizeable share of the bound


def test_flag_rule_edges():
    # A = 0: reference and magnitude vanish and the bound is its subnormal term 2 K N 2^-126
    M, N, K = 4, 8, 16
    Ab = np.zeros((M, K), dtype=np.uint16)
    Wb = _bf16_round(np.ones((N, K), np.float32))
    b = 2.0 * K * N * 2.0 ** -126
    rowsum = np.array([b, 2 * b, np.nan, -np.inf])
    v = oracle.abft_verify(rowsum, Ab, Wb, tol_scale=1.0)
    assert np.all(v["bound"] == b)
    assert list(v["flag"]) == [0, 1, 1, 1]  # equality passes; NaN and infinities flag
    v = oracle.abft_verify(rowsum, Ab, Wb, tol_scale=2.0)
    assert list(v["flag"]) == [0, 0, 1, 1]


def test_column_identity_and_planted_weight_fault():
    # 1^T (A W^T) = (1^T A) W^T exactly on integers; a fault in W's row j (the GEMM reads
    # W' = W + delta e_(j,k), the check uses W) moves column j's residual by delta sum_i A[i, k]
    M, N, K = 12, 10, 18
    A, W, Ab, Wb = _int_operands(M, N, K, 7, lo=-8, hi=8)
    colsum = oracle.abft_product(Ab, Wb).sum(axis=0)
    brute = [sum(int(A[i, k]) * int(W[j, k]) for i in range(M) for k in range(K)) for j in range(N)]
    assert list(colsum) == brute
    v = oracle.abft_verify_cols(colsum, Ab, Wb)
    assert v["n_flagged"] == 0 and np.all(v["residual"] == 0)
    j, k, delta = 4, 9, 5
    Wf = W.copy()
    Wf[j, k] += delta
    colsum_f = oracle.abft_product(Ab, _bf16_bits(Wf.astype(np.float32))).sum(axis=0)
    v = oracle.abft_verify_cols(colsum_f, Ab, Wb)
    expect = np.zeros(N)
    expect[j] = delta * int(A[:, k].sum())
    assert np.array_equal(v["residual"], expect)
    # the row check sees the same fault spread over every row: delta A[i, k] on row i
    vr = oracle.abft_verify(oracle.abft_product(Ab, _bf16_bits(Wf.astype(np.float32))).sum(axis=1), Ab, Wb)
    assert np.array_equal(vr["residual"], delta * A[:, k].astype(float))


@pytest.mark.parametrize("mode", ["rn", "trunc", "block16"])
def test_column_bound_covers_float32_accumulation(mode):
    M, N, K = 32, 8, 512
    rng = np.random.default_rng(8)
    A32 = (rng.uniform(0.5, 1.0, (M, K)) * 2.0 ** -rng.integers(0, 12, (M, K))).astype(np.float32)
    W32 = (rng.uniform(0.5, 1.0, (N, K)) * 2.0 ** -rng.integers(0, 12, (N, K))).astype(np.float32)
    A32[:, 0], W32[:, 0] = 2.0 ** 10, 2.0 ** 4
    Ab, Wb = _bf16_round(A32), _bf16_round(W32)
    acc = _emulate_fp32(oracle.bf16_to_f64(Ab), oracle.bf16_to_f64(Wb), mode)
    v = oracle.abft_verify_cols(acc.sum(axis=0), Ab, Wb)
    assert v["n_flagged"] == 0
    assert np.max(np.abs(v["residual"]) / v["bound"]) <= 1.0


# ---------------------------------------------------------------- weight-gradient configuration
# dW = dY^T X with dY [T, N] and X [T, K] token-major; the row + column configuration covers it
# ([AEGIS] method section 2).

def test_wgrad_product_and_both_sides_brute_force():
    T, N, K = 9, 7, 12
    rng = np.random.default_rng(21)
    dY, X = rng.integers(-9, 10, size=(T, N)), rng.integers(-9, 10, size=(T, K))
    dYb, Xb = _bf16_bits(dY.astype(np.float32)), _bf16_bits(X.astype(np.float32))
    brute = [[sum(int(dY[t, n]) * int(X[t, k]) for t in range(T)) for k in range(K)] for n in range(N)]
    dW = oracle.wgrad_product(dYb, Xb)
    assert dW.tolist() == brute
    ref = oracle.wgrad_reference(dYb, Xb)
    assert ref["row_ref"].tolist() == [sum(r) for r in brute]
    assert ref["col_ref"].tolist() == [sum(brute[n][k] for n in range(N)) for k in range(K)]
    assert ref["row_mag"].tolist() == [sum(abs(int(dY[t, n])) * sum(abs(int(x)) for x in X[t]) for t in range(T))
                                       for n in range(N)]
    assert ref["col_mag"].tolist() == [sum(sum(abs(int(y)) for y in dY[t]) * abs(int(X[t, k])) for t in range(T))
                                       for k in range(K)]
    v = oracle.wgrad_verify(dW.sum(axis=1), dW.sum(axis=0), dYb, Xb)
    assert v["n_flagged"] == 0 and v["n_flagged_col"] == 0
    assert np.all(v["residual"] == 0) and np.all(v["residual_col"] == 0)


def test_wgrad_single_token_is_an_outer_product():
    rng = np.random.default_rng(22)
    dY, X = rng.integers(-5, 6, size=(1, 6)), rng.integers(-5, 6, size=(1, 10))
    dYb, Xb = _bf16_bits(dY.astype(np.float32)), _bf16_bits(X.astype(np.float32))
    assert np.array_equal(oracle.wgrad_product(dYb, Xb), np.outer(dY[0], X[0]).astype(float))


@pytest.mark.parametrize("operand", ["dY", "X"])
def test_wgrad_planted_fault_closed_form(operand):
    # the product reads a faulty operand, the check the clean one: a change delta at (t, j) moves
    # dY fault (t, n): row n by delta sum_k X[t, k], column k by delta X[t, k]
    # X fault (t, k): column k by delta sum_n dY[t, n], row n by delta dY[t, n]
    T, N, K = 11, 8, 16
    rng = np.random.default_rng(23)
    dY, X = rng.integers(-8, 9, size=(T, N)), rng.integers(-8, 9, size=(T, K))
    dYb, Xb = _bf16_bits(dY.astype(np.float32)), _bf16_bits(X.astype(np.float32))
    t, delta = 5, 3
    if operand == "dY":
        n = 6
        dYf = dY.copy()
        dYf[t, n] += delta
        dW = oracle.wgrad_product(_bf16_bits(dYf.astype(np.float32)), Xb)
        er = np.zeros(N)
        er[n] = delta * X[t].sum()
        ec = np.zeros(K)
        ec[:] = delta * X[t]
    else:
        k = 13
        Xf = X.copy()
        Xf[t, k] += delta
        dW = oracle.wgrad_product(dYb, _bf16_bits(Xf.astype(np.float32)))
        er = (delta * dY[t]).astype(float)
        ec = np.zeros(K)
        ec[k] = delta * dY[t].sum()
    v = oracle.wgrad_verify(dW.sum(axis=1), dW.sum(axis=0), dYb, Xb)
    assert np.array_equal(v["residual"], er)
    assert np.array_equal(v["residual_col"], ec)


@pytest.mark.parametrize("mode", ["rn", "trunc", "block16"])
def test_wgrad_bound_covers_float32_accumulation(mode):
    # accumulation over the tokens, emulated on dW = (dY^T)(X^T)^T; both sides within their bounds
    T, N, K = 512, 16, 24
    rng = np.random.default_rng(24)
    dY32 = (rng.uniform(0.5, 1.0, (T, N)) * 2.0 ** -rng.integers(0, 12, (T, N))).astype(np.float32)
    X32 = (rng.uniform(0.5, 1.0, (T, K)) * 2.0 ** -rng.integers(0, 12, (T, K))).astype(np.float32)
    dY32[0], X32[0] = 2.0 ** 9, 2.0 ** 5
    dYb, Xb = _bf16_round(dY32), _bf16_round(X32)
    acc = _emulate_fp32(oracle.bf16_to_f64(dYb).T.copy(), oracle.bf16_to_f64(Xb).T.copy(), mode)
    v = oracle.wgrad_verify(acc.sum(axis=1), acc.sum(axis=0), dYb, Xb)
    assert v["n_flagged"] == 0 and v["n_flagged_col"] == 0
    assert np.max(np.abs(v["residual"]) / v["bound"]) <= 1.0
    assert np.max(np.abs(v["residual_col"]) / v["bound_col"]) <= 1.0
    ref = oracle.wgrad_reference(dYb, Xb)  # not vacuous: about T 2^-22 of the magnitude
    assert np.all(v["bound"] <= 1.01 * T * 2.0 ** -22 * ref["row_mag"] + 1e-30)
    if mode == "trunc":
        assert np.max(np.abs(v["residual"]) / v["bound"]) > 0.05


def test_wgrad_flag_rule_edges():
    T, N, K = 3, 8, 16
    dYb = np.zeros((T, N), dtype=np.uint16)
    Xb = _bf16_round(np.ones((T, K), np.float32))
    b, bc = 2.0 * T * K * 2.0 ** -126, 2.0 * T * N * 2.0 ** -126
    rowsum = np.array([b, 2 * b, np.nan, -np.inf, 0, 0, 0, 0])
    v = oracle.wgrad_verify(rowsum, np.zeros(K), dYb, Xb)
    assert np.all(v["bound"] == b) and np.all(v["bound_col"] == bc)
    assert list(v["flag"]) == [0, 1, 1, 1, 0, 0, 0, 0] and v["n_flagged_col"] == 0
    assert "residual_col" not in oracle.wgrad_verify(rowsum, None, dYb, Xb)


# ---------------------------------------------------------------- replay context and replay

def test_capture_index_order_cap_and_count():
    idx, n = oracle.capture_index(np.array([0, 1, 0, 1, 1, 0, 1], np.uint8), 3)
    assert idx.tolist() == [1, 3, 4] and n == 4
    idx, n = oracle.capture_index(np.zeros(5, np.uint8), 4)
    assert idx.tolist() == [] and n == 0


def test_capture_copies_rows_and_columns_by_hand():
    M, N, K = 5, 6, 4
    A = np.arange(M * K, dtype=np.uint16).reshape(M, K)
    Wb = (1000 + np.arange(N * K, dtype=np.uint16)).reshape(N, K)
    C = (5000 + np.arange(M * N, dtype=np.uint16)).reshape(M, N)
    cap = oracle.abft_capture(np.array([0, 1, 0, 0, 1], np.uint8), np.array([1, 0, 0, 1, 0, 1], np.uint8),
                              A, Wb, C, cap_rows=4, cap_cols=2)
    assert cap["n_rows"] == 2 and cap["n_cols"] == 3
    assert cap["row_idx"].tolist() == [1, 4] and cap["col_idx"].tolist() == [0, 3]
    assert cap["row_A"].tolist() == [[4, 5, 6, 7], [16, 17, 18, 19]]
    assert cap["row_C"].tolist() == [[5006 + j for j in range(6)], [5024 + j for j in range(6)]]
    assert cap["col_W"].tolist() == [[1000, 1001, 1002, 1003], [1012, 1013, 1014, 1015]]
    assert cap["col_C"].tolist() == [[5000 + 6 * i for i in range(5)], [5003 + 6 * i for i in range(5)]]
    # the weight-gradient form: dY's and X's columns, dW's rows and columns
    T = 3
    dY = np.arange(T * N, dtype=np.uint16).reshape(T, N)
    X = (100 + np.arange(T * K, dtype=np.uint16)).reshape(T, K)
    dW = (7000 + np.arange(N * K, dtype=np.uint16)).reshape(N, K)
    w = oracle.wgrad_capture(np.array([0, 0, 1, 0, 0, 1], np.uint8), np.array([0, 1, 0, 0], np.uint8),
                             dY, X, dW, cap_rows=1, cap_cols=4)
    assert w["n_rows"] == 2 and w["row_idx"].tolist() == [2] and w["n_cols"] == 1 and w["col_idx"].tolist() == [1]
    assert w["row_dY"].tolist() == [[2, 8, 14]] and w["row_dW"].tolist() == [[7008, 7009, 7010, 7011]]
    assert w["col_X"].tolist() == [[101, 105, 109]]
    assert w["col_dW"].tolist() == [[7001 + 4 * n for n in range(N)]]


def test_replay_consistency_exact_and_planted():
    # integer operands: every product and sum is exact, so C (bf16 of small integers) equals the
    # exact product; one element moved by more than the rounding bound is the only one flagged
    M, N, K = 4, 16, 32
    A, W, Ab, Wb = _int_operands(M, N, K, 31, lo=-3, hi=3)
    C = (A @ W.T).astype(np.float32)
    Cb = _bf16_bits(C)
    assert oracle.abft_replay_rows(Ab, Wb, Cb).tolist() == [0, 0, 0, 0]
    bad = C.copy()
    bad[2, 7] += 64.0  # |C| <= 288: exact in bf16 after the move, far beyond the bound
    assert oracle.abft_replay_rows(Ab, Wb, _bf16_bits(bad)).tolist() == [0, 0, 1, 0]


@pytest.mark.parametrize("mode", ["rn", "trunc", "block16"])
def test_replay_consistency_covers_float32_accumulation(mode):
    # a correct computation (float32 accumulation in any order, then bf16 rounding) is consistent
    # everywhere; a value two bounds away is not
    M, N, K = 6, 24, 512
    rng = np.random.default_rng(32)
    A32 = (rng.uniform(0.5, 1.0, (M, K)) * 2.0 ** -rng.integers(0, 12, (M, K))).astype(np.float32)
    W32 = (rng.uniform(0.5, 1.0, (N, K)) * 2.0 ** -rng.integers(0, 12, (N, K))).astype(np.float32)
    Ab, Wb = _bf16_round(A32), _bf16_round(W32)
    acc = _emulate_fp32(oracle.bf16_to_f64(Ab), oracle.bf16_to_f64(Wb), mode)
    Cb = _bf16_round(acc.astype(np.float32))
    assert np.all(oracle.abft_replay_rows(Ab, Wb, Cb) == 0)
    exact = oracle.abft_product(Ab, Wb)
    shifted = _bf16_round((exact * (1.0 + 2.0 ** -5)).astype(np.float32))  # 2^-5: four times the bf16 step
    assert np.all(oracle.abft_replay_rows(Ab, Wb, shifted) == N)


def test_wgrad_replay_pairs_flags_only_the_planted_element():
    T, N, K = 10, 8, 12
    rng = np.random.default_rng(33)
    dY, X = rng.integers(-4, 5, size=(T, N)), rng.integers(-4, 5, size=(T, K))
    dYb, Xb = _bf16_bits(dY.astype(np.float32)), _bf16_bits(X.astype(np.float32))
    dW = (dY.T @ X).astype(np.float32)
    dW[5, 3] += 32.0
    cap = oracle.wgrad_capture(np.array([0, 1, 0, 0, 0, 1, 0, 0], np.uint8),
                               np.array([0, 0, 0, 1, 0, 0, 0, 0, 0, 1, 0, 0], np.uint8),
                               dYb, Xb, _bf16_bits(dW), cap_rows=2, cap_cols=2)
    assert oracle.wgrad_replay_pairs(cap).tolist() == [[0, 0], [1, 0]]


def test_forward_replay_pairs_flags_only_the_planted_element():
    M, N, K = 9, 12, 10
    A, W, Ab, Wb = _int_operands(M, N, K, 34, lo=-4, hi=4)
    C = (A @ W.T).astype(np.float32)
    C[2, 7] += 64.0
    cap = oracle.abft_capture(np.isin(np.arange(M), [2, 5]), np.isin(np.arange(N), [3, 7]), Ab, Wb, _bf16_bits(C),
                              cap_rows=2, cap_cols=2)
    assert oracle.abft_replay_pairs(cap).tolist() == [[0, 1], [0, 0]]
