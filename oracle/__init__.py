"""CPU oracle for the replica-integrity scan.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg do.  It shares no code with the CUDA path.

Sources (web pages on silent data corruption):
  [AWS]   "Detecting and recovering from silent data corruption on Amazon
          SageMaker HyperPod" (AWS Machine Learning Blog).
  [AEGIS] "Safeguarding LLM Training at Scale: Online SDC Detection and
          Insights from 35 Million GPU Hours" (review page).

The GEMM checksum and attention-invariant functions at the end are plain numpy
in float64; their parity with the tensor-core kernels is up to the rounding
bounds they state.

The element loops live in ``sdc_oracle.c`` (plain scalar C, compiled with gcc
on first use); the vote and the exact rounding of the sum of squares are plain
Python.  Every function takes host numpy arrays.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from collections import Counter
from concurrent.futures import ThreadPoolExecutor
from fractions import Fraction

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# dtype codes of the oracle's C file (its own numbering)
DTYPE_CODES = {"f32": 1, "bf16": 2, "f16": 3}
ESIZE = {"f32": 4, "bf16": 2, "f16": 2}
_QMIN = -149
_NBINS = 270
FLT_MAX = 3.4028234663852886e38

_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile sdc_oracle.c into oracle/_build/liboracle.so (gcc, -O2).

    ``-ffp-contract=off`` keeps every float operation a separately rounded
    IEEE operation (no fused multiply-add), as the average's definition needs.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64p = ctypes.POINTER(ctypes.c_uint64)
            lib.oracle_fingerprint.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32,
                                               ctypes.c_uint64, u64p]
            lib.oracle_fingerprint.restype = ctypes.c_int
            lib.oracle_xorsum.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, u64p]
            lib.oracle_xorsum.restype = ctypes.c_int
            lib.oracle_grad_stats.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32,
                                              u64p, u64p]
            lib.oracle_grad_stats.restype = ctypes.c_int
            lib.oracle_average.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint32,
                                           ctypes.c_uint64, ctypes.c_uint32, ctypes.c_void_p]
            lib.oracle_average.restype = ctypes.c_int
            fl = ctypes.c_float
            lib.oracle_adamw.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint32, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_uint64, fl, ctypes.c_int, fl, fl, fl, fl, fl,
                                         fl, fl]
            lib.oracle_adamw.restype = ctypes.c_int
            lib.oracle_round_f32.argtypes = [ctypes.c_float, ctypes.c_uint32]
            lib.oracle_round_f32.restype = ctypes.c_uint32
            _lib = lib
    return _lib


def _as_bytes(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _slices(numel: int, threads: int, min_slice: int = 1 << 22):
    """Consecutive element slices [lo, hi) used to spread one loop over threads."""
    if threads <= 1 or numel <= min_slice:
        return [(0, numel)]
    n = min(threads * 4, max(1, numel // min_slice))
    step = -(-numel // n)
    return [(lo, min(numel, lo + step)) for lo in range(0, numel, step)]


# --------------------------------------------------------------------------
# Fingerprint  ([AWS] "Compare by fingerprint")
# --------------------------------------------------------------------------
def fingerprint(a: np.ndarray, threads: int = 1) -> tuple[int, int]:
    """(S, W) of one tensor: S = sum of widened raw bits, W = sum of (index+1)*bits.

    Both mod 2^64, returned as Python ints in [0, 2^64).  ``a`` is any
    contiguous numpy array; its itemsize selects the bit view.  With
    ``threads > 1`` the tensor is walked in consecutive slices (each weighted
    by its global index, as the page's chunk loop does) on a thread pool and
    the slices' sums are added mod 2^64.
    """
    lib = _load()
    a = _as_bytes(a)
    esize = a.itemsize
    numel = a.size
    base = _ptr(a)

    def run(lo_hi):
        lo, hi = lo_hi
        out = (ctypes.c_uint64 * 2)()
        rc = lib.oracle_fingerprint(base + lo * esize, hi - lo, esize, lo, out)
        if rc != 0:
            raise ValueError(f"bad element size {esize}")
        return out[0], out[1]

    parts = _map(run, _slices(numel, threads), threads)
    s = sum(p[0] for p in parts) % (1 << 64)
    w = sum(p[1] for p in parts) % (1 << 64)
    return s, w


def xorsum(a: np.ndarray, threads: int = 1) -> int:
    """XOR of every element's raw bits, zero-extended to 64 bits ([AEGIS] sec. 4)."""
    lib = _load()
    a = _as_bytes(a)
    esize = a.itemsize
    base = _ptr(a)

    def run(lo_hi):
        lo, hi = lo_hi
        out = ctypes.c_uint64()
        if lib.oracle_xorsum(base + lo * esize, hi - lo, esize, ctypes.byref(out)) != 0:
            raise ValueError(f"bad element size {esize}")
        return out.value

    x = 0
    for p in _map(run, _slices(a.size, threads), threads):
        x ^= p
    return x


def xorsum_compare(a: list[int], b: list[int]) -> tuple[list[int], list[int]]:
    """Pairwise compare of two xorsum lists: (mismatch flags, a XOR b)."""
    mism = [1 if x != y else 0 for x, y in zip(a, b)]
    diff = [x ^ y for x, y in zip(a, b)]
    return mism, diff


def _map(fn, items, threads):
    if threads <= 1 or len(items) == 1:
        return [fn(it) for it in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))


# --------------------------------------------------------------------------
# Gradient statistics  ([AWS] "Check 1: NaN/Inf gradients, before and after
# the all-reduce"; "Decide what the alarm means")
# --------------------------------------------------------------------------
def exact_sum_from_bins(bins: np.ndarray) -> float:
    """Correctly rounded double of sum_b bins[b] * 4^(b + QMIN).

    ``bins`` is a (NBINS, 2) uint64 array of 128-bit integers (lo, hi).  The
    sum is formed exactly with rationals and rounded once (Fraction -> float
    rounds to nearest, ties to even).
    """
    total = Fraction(0)
    for b in range(_NBINS):
        v = int(bins[b, 0]) | (int(bins[b, 1]) << 64)
        if v:
            total += Fraction(v) * Fraction(2) ** (2 * (b + _QMIN))
    return float(total)


def grad_stats(a: np.ndarray, dtype: str, threads: int = 1) -> dict:
    """Non-finite counts and exact sum of squares of one gradient buffer.

    Returns n_nan, n_inf, n_big (finite, x^2 > FLT_MAX), n_elems,
    sumsq_finite (exact sum of x^2 over finite x, rounded once to double),
    norm (NaN if any NaN, else +Inf if any Inf, else sqrt(sumsq_finite)) and
    nonfinite_fp32 (the page's float32 flag: any NaN/Inf, or a squared norm
    above FLT_MAX, i.e. a norm above ~1.8e19).
    ``a`` holds the raw elements (uint16 for bf16/f16, float32/uint32 for f32).
    """
    if np.asarray(a).itemsize != ESIZE[dtype]:
        raise ValueError("element size does not match dtype")
    return grad_stats_multi([a], [dtype], threads)


def finish_stats(n_nan: int, n_inf: int, n_big: int, n_elems: int, sumsq: float) -> dict:
    """Derived fields of a stats record (norm with IEEE propagation, fp32 flag)."""
    if n_nan:
        norm = math.nan
    elif n_inf:
        norm = math.inf
    else:
        norm = math.sqrt(sumsq)
    nonfinite = 1 if (n_nan or n_inf or sumsq > FLT_MAX) else 0
    return {"n_nan": n_nan, "n_inf": n_inf, "n_big": n_big, "n_elems": n_elems,
            "sumsq_finite": sumsq, "norm": norm, "nonfinite_fp32": nonfinite}


def grad_stats_multi(arrays: list[np.ndarray], dtypes: list[str], threads: int = 1) -> dict:
    """Stats of one replica made of several tensors, summed exactly once.

    All tensors' squares go into one set of exponent bins, so the result is
    the exact sum over every finite element of every tensor, rounded once.
    """
    lib = _load()
    counts = np.zeros(3, dtype=np.uint64)
    acc = [0] * _NBINS
    n = 0
    lock = threading.Lock()

    def run(item):
        a, dt, lo, hi = item
        c = np.zeros(3, dtype=np.uint64)
        bins = np.zeros((_NBINS, 2), dtype=np.uint64)
        lib.oracle_grad_stats(_ptr(a) + lo * a.itemsize, hi - lo, DTYPE_CODES[dt],
                              c.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                              bins.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)))
        with lock:
            counts[:] += c
            for b in np.nonzero(bins[:, 0] | bins[:, 1])[0]:
                acc[b] += int(bins[b, 0]) | (int(bins[b, 1]) << 64)

    items = []
    for a, dt in zip(arrays, dtypes):
        a = _as_bytes(a)
        n += a.size
        for lo, hi in _slices(a.size, threads):
            items.append((a, dt, lo, hi))
    _map(run, items, threads)
    merged = np.zeros((_NBINS, 2), dtype=np.uint64)
    for b in range(_NBINS):
        merged[b, 0] = acc[b] & ((1 << 64) - 1)
        merged[b, 1] = acc[b] >> 64
    return finish_stats(int(counts[0]), int(counts[1]), int(counts[2]), n,
                        exact_sum_from_bins(merged))


# --------------------------------------------------------------------------
# Average of local gradients  ([AWS] "Step 1: Detect", worked example)
# --------------------------------------------------------------------------
def average(bufs: list[np.ndarray], dtype: str, threads: int = 1) -> np.ndarray:
    """float32 sum in buffer order, / n, rounded to dtype (ties to even); NaN canonical."""
    lib = _load()
    code = DTYPE_CODES[dtype]
    bufs = [_as_bytes(b) for b in bufs]
    numel = bufs[0].size
    for b in bufs:
        if b.size != numel or b.itemsize != ESIZE[dtype]:
            raise ValueError("buffers disagree in size")
    out = np.empty(numel, dtype=np.uint32 if dtype == "f32" else np.uint16)
    es = ESIZE[dtype]

    def run(lo_hi):
        lo, hi = lo_hi
        ptrs = (ctypes.c_void_p * len(bufs))(*[_ptr(b) + lo * es for b in bufs])
        rc = lib.oracle_average(ptrs, len(bufs), hi - lo, code, _ptr(out) + lo * es)
        if rc != 0:
            raise ValueError("bad arguments")

    _map(run, _slices(numel, threads), threads)
    return out


def round_f32(x: float, dtype: str) -> int:
    """Bits of float32 x rounded to bf16/f16 by the oracle's own rounding."""
    return int(_load().oracle_round_f32(ctypes.c_float(x), DTYPE_CODES[dtype]))


# --------------------------------------------------------------------------
# Strict-majority vote  ([AWS] "Check 3: Weight fingerprints, after the
# optimizer step")
# --------------------------------------------------------------------------
SUSPECT_AGREE = -1
SUSPECT_SEVERAL = -2
SUSPECT_NO_MAJORITY = -3


def vote(table) -> tuple[list[int], list[int], dict]:
    """Per-tensor vote over R replicas' fingerprints.

    ``table[r][k]`` is replica r's fingerprint (a tuple) of tensor k.  For each
    tensor whose copies do not all agree, the most common fingerprint is a
    strict majority only if it is held by more than half of the R copies; a
    replica is a suspect when its copy differs from that majority.  Returns
    (suspect, mask, summary):
      suspect[k]: -1 all agree, r if exactly replica r differs, -2 if several
                  differ from a majority, -3 if there is no strict majority;
      mask[k]:    bit r set when replica r differs from the majority
                  (0 when all agree or there is no majority);
      summary:    diverged (any tensor differs), no_majority (some differing
                  tensor lacks a strict majority), suspect_mask (union of the
                  masks of tensors that have a majority).
    """
    R = len(table)
    T = len(table[0]) if R else 0
    suspect = [SUSPECT_AGREE] * T
    mask = [0] * T
    diverged = False
    no_majority = False
    union = 0
    for k in range(T):
        copies = [tuple(table[r][k]) for r in range(R)]
        if all(c == copies[0] for c in copies):
            continue
        diverged = True
        value, count = Counter(copies).most_common(1)[0]
        if 2 * count <= R:
            suspect[k] = SUSPECT_NO_MAJORITY
            no_majority = True
            continue
        odd = [r for r, c in enumerate(copies) if c != value]
        m = 0
        for r in odd:
            m |= 1 << r
        mask[k] = m
        suspect[k] = odd[0] if len(odd) == 1 else SUSPECT_SEVERAL
        union |= m
    return suspect, mask, {"diverged": int(diverged), "no_majority": int(no_majority),
                           "suspect_mask": union}


def pages_verdict(summary: dict) -> dict:
    """The page's result dict from a vote summary.

    No divergence -> {"diverged": False, "suspects": []}; any differing tensor
    without a strict majority -> {"diverged": True, "suspects": None};
    otherwise the sorted replicas that differ from a majority somewhere.
    """
    if not summary["diverged"]:
        return {"diverged": False, "suspects": []}
    if summary["no_majority"]:
        return {"diverged": True, "suspects": None}
    m = summary["suspect_mask"]
    return {"diverged": True, "suspects": [r for r in range(64) if (m >> r) & 1]}


# --------------------------------------------------------------------------
# Ring replay audit  ([AWS] "Check 2: Ring replay, before the optimizer step")
# --------------------------------------------------------------------------
def ring_pairs(table, offset: int) -> list[tuple[int, int]]:
    """Mismatched (target, replayer) pairs of a ring audit table.

    ``table[r]`` is rank r's pair of rows (own result, replay of its target);
    rank r replays rank (r + offset) % n.  A pair mismatches when the target's
    own result differs from the replayer's replay.  Listed by replayer.
    """
    n = len(table)
    out = []
    for r in range(n):
        t = (r + offset) % n
        if list(table[t][0]) != list(table[r][1]):
            out.append((t, r))
    return out


def localize(pairs: list[tuple[int, int]]) -> tuple[list[int], list[tuple[int, int]]]:
    """Culprits (ranks counted in two or more mismatched pairs) and the pairs touching none of them."""
    hits = Counter(x for p in pairs for x in p)
    culprits = sorted(r for r, c in hits.items() if c >= 2)
    ambiguous = [p for p in pairs if not (set(p) & set(culprits))]
    return culprits, ambiguous


# --------------------------------------------------------------------------
# Clip + AdamW step  ([AWS] "Use case: Testing the checks on SageMaker
# HyperPod" hyperparameters; `train()` clip, reduced-gradient gate and step)
# --------------------------------------------------------------------------
def adamw_scalars(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, step: int) -> dict:
    """float32 scalars of one AdamW step: each formed in double from the float32 inputs, rounded once."""
    f = lambda x: float(np.float32(x))
    lr, beta1, beta2, eps, wd = f(lr), f(beta1), f(beta2), f(eps), f(weight_decay)
    return {"decay": f(1.0 - lr * wd), "omb1": f(1.0 - beta1), "beta2": beta2, "omb2": f(1.0 - beta2),
            "bc2s": f(math.sqrt(1.0 - math.pow(beta2, step))), "eps": eps,
            "step_size": f(lr / (1.0 - math.pow(beta1, step)))}


def clip_coef(norm: float, max_norm: float) -> float:
    """clip_grad_norm_'s coefficient in float32: min(1, max_norm / (norm + 1e-6))."""
    n32 = np.float32(norm)
    c = np.float32(np.float32(max_norm) / np.float32(n32 + np.float32(1e-6)))
    return float(min(c, np.float32(1.0)))


def adamw_step(p: np.ndarray, grad: np.ndarray, gdtype: str, m: np.ndarray, v: np.ndarray, hp: dict,
               post_stats: dict | None) -> bool:
    """One gated, clipped AdamW step on float32 host arrays, in place.

    ``hp``: lr, beta1, beta2, eps, weight_decay, max_grad_norm, step, clip.  When
    ``post_stats`` (the reduced gradient's stats) raise the float32 alarm, nothing is
    updated and False is returned, as the page's train() skips the step.
    """
    if post_stats is not None and post_stats["nonfinite_fp32"]:
        return False
    k = adamw_scalars(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], hp["step"])
    use = 1 if (hp.get("clip") and post_stats is not None) else 0
    coef = clip_coef(post_stats["norm"], hp["max_grad_norm"]) if use else 1.0
    for a in (p, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    g = np.ascontiguousarray(grad)
    rc = _load().oracle_adamw(p.ctypes.data, g.ctypes.data, DTYPE_CODES[gdtype], m.ctypes.data, v.ctypes.data,
                              p.size, coef, use, k["decay"], k["omb1"], k["beta2"], k["omb2"], k["bc2s"], k["eps"],
                              k["step_size"])
    if rc != 0:
        raise ValueError("bad grad dtype")
    return True


# --------------------------------------------------------------------------
# GEMM checksum  ([AEGIS] method section 2: (AB)1 against A(B1), the checksum
# taken from the float32 accumulator before the bfloat16 output is rounded)
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64, exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def abft_product(A_bits: np.ndarray, W_bits: np.ndarray) -> np.ndarray:
    """C = A . W^T in float64 for bf16 A [M, K] and W [N, K] (K contiguous in both).

    Every product of two bf16 values is exact in float64; the K-term sums round at
    most K * 2^-53 of sum_k |a| |w|, far below the float32 accumulation error the
    check bounds."""
    return bf16_to_f64(A_bits) @ bf16_to_f64(W_bits).T


def abft_row_checksum(C: np.ndarray) -> np.ndarray:
    """(AB)1: each output row summed."""
    return C.sum(axis=1)


def abft_reference(A_bits: np.ndarray, W_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """A(B1) and the magnitude sum_k |A[i,k]| sum_j |W[j,k]| of each row, float64.

    B1 for C = A W^T is W^T 1: the column sums of W over its N rows."""
    A = bf16_to_f64(A_bits)
    W = bf16_to_f64(W_bits)
    w1 = W.sum(axis=0)
    wabs = np.abs(W).sum(axis=0)
    return A @ w1, np.abs(A) @ wabs


def abft_bound(mag: np.ndarray, N: int, K: int) -> np.ndarray:
    """Rounding bound of a checksum of N outputs taken from their float32 accumulators
    (N: the columns a row checksum sums, or the rows a column checksum sums), against
    exact check sums.

    Each of the K float32 accumulation steps of one output may lose up to two
    units in the last place of its partial sum (g = K 2^-22 per output to first
    order, g^2 beyond it); subnormals flushed to zero lose 2^-126 per product and
    per step.  The check's own sums are taken as exact: here they are float64,
    whose rounding (below (N + K) 2^-53 of the magnitude) is far under one float32
    unit of the bound.  A check that carries its sums in less precision adds its
    own term on top."""
    g = K * 2.0 ** -22
    return g * (1.0 + g) * np.asarray(mag, dtype=np.float64) + 2.0 * K * N * 2.0 ** -126


def abft_reference_cols(A_bits: np.ndarray, W_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(1^T A) W^T and the magnitude sum_k (sum_i |A[i,k]|) |W[j,k]| of each output column, float64:
    the column side of the check (the page's row + column configuration)."""
    A = bf16_to_f64(A_bits)
    W = bf16_to_f64(W_bits)
    return W @ A.sum(axis=0), np.abs(W) @ np.abs(A).sum(axis=0)


def abft_verify_cols(colsum: np.ndarray, A_bits: np.ndarray, W_bits: np.ndarray, tol_scale: float = 1.0) -> dict:
    """The column check: residual = 1^T C (accumulator) - (1^T A) W^T per column, its bound (the
    row bound with the M summed rows in place of the N summed columns), the column flags."""
    M, K = A_bits.shape
    ref, mag = abft_reference_cols(A_bits, W_bits)
    residual = np.asarray(colsum, dtype=np.float64) - ref
    bound = abft_bound(mag, M, K)
    with np.errstate(invalid="ignore"):
        flag = ~(np.abs(residual) <= tol_scale * bound)
    return {"residual": residual, "bound": bound, "flag": flag.astype(np.uint8), "n_flagged": int(flag.sum())}


def abft_verify(rowsum: np.ndarray, A_bits: np.ndarray, W_bits: np.ndarray, tol_scale: float = 1.0) -> dict:
    """The check of one GEMM: residual = checksum - A(W^T 1), the bound, and the
    row flags (a row is flagged unless |residual| <= tol_scale * bound, so a NaN
    residual flags)."""
    M, K = A_bits.shape
    N = W_bits.shape[0]
    ref, mag = abft_reference(A_bits, W_bits)
    residual = np.asarray(rowsum, dtype=np.float64) - ref
    bound = abft_bound(mag, N, K)
    with np.errstate(invalid="ignore"):
        flag = ~(np.abs(residual) <= tol_scale * bound)
    return {"residual": residual, "bound": bound, "flag": flag.astype(np.uint8), "n_flagged": int(flag.sum())}


# --------------------------------------------------------------------------
# Weight-gradient configuration  ([AEGIS] method section 2: the row
# configuration leaves wgrad partly uncovered, the row + column configuration
# covers every matmul class, wgrad included).  A linear layer's weight gradient
# is dW = dY^T X, with the output gradient dY [T, N] and the layer's input
# X [T, K] held token-major, as the backward pass has them; the contraction
# runs over the T tokens.
# --------------------------------------------------------------------------
def wgrad_product(dY_bits: np.ndarray, X_bits: np.ndarray) -> np.ndarray:
    """dW = dY^T X in float64 for bf16 dY [T, N] and X [T, K]: dW [N, K]."""
    return bf16_to_f64(dY_bits).T @ bf16_to_f64(X_bits)


def wgrad_reference(dY_bits: np.ndarray, X_bits: np.ndarray) -> dict:
    """The two sides of the check of dW = dY^T X, float64.

    Rows: dW 1 = dY^T (X 1), and the magnitude sum_t |dY[t, n]| sum_k |X[t, k]|.
    Columns: 1^T dW = (1^T dY^T) X = (dY 1)^T X, and the magnitude
    sum_t (sum_n |dY[t, n]|) |X[t, k]|."""
    dY = bf16_to_f64(dY_bits)
    X = bf16_to_f64(X_bits)
    r, ra = X.sum(axis=1), np.abs(X).sum(axis=1)    # X 1 and |X| 1, one per token
    q, qa = dY.sum(axis=1), np.abs(dY).sum(axis=1)  # dY 1 and |dY| 1
    return {"row_ref": dY.T @ r, "row_mag": np.abs(dY).T @ ra, "col_ref": X.T @ q, "col_mag": np.abs(X).T @ qa}


def wgrad_verify(rowsum: np.ndarray, colsum, dY_bits: np.ndarray, X_bits: np.ndarray,
                 tol_scale: float = 1.0) -> dict:
    """The check of one weight-gradient product: per output row n, residual = the
    accumulator checksum - dY^T (X 1), bound over the K outputs the row sums with a
    contraction of T; per output column (colsum given), the same over the N rows.
    A row or column flags unless |residual| <= tol_scale * bound (NaN flags)."""
    T, N = dY_bits.shape
    K = X_bits.shape[1]
    ref = wgrad_reference(dY_bits, X_bits)
    out = {}
    sides = [("", rowsum, ref["row_ref"], ref["row_mag"], K)]
    if colsum is not None:
        sides.append(("_col", colsum, ref["col_ref"], ref["col_mag"], N))
    for tag, got, want, mag, n_sum in sides:
        residual = np.asarray(got, dtype=np.float64) - want
        bound = abft_bound(mag, n_sum, T)
        with np.errstate(invalid="ignore"):
            flag = ~(np.abs(residual) <= tol_scale * bound)
        out.update({"residual" + tag: residual, "bound" + tag: bound, "flag" + tag: flag.astype(np.uint8),
                    "n_flagged" + tag: int(flag.sum())})
    return out


# --------------------------------------------------------------------------
# Replay context and replay  ([AEGIS] method sections 1 and 2: when a check
# fires, the sensor packs its evidence and the least context a replay needs
# into a vTask; a verifier replays it off the critical path and confirms.  For
# the forward product the context is the flagged row of A and the output row;
# for wgrad, A's rows, B's columns and the matching results.)
# --------------------------------------------------------------------------
def capture_index(flag: np.ndarray, cap: int) -> tuple[np.ndarray, int]:
    """The flagged positions in increasing order, at most cap of them, and how many were flagged."""
    idx = np.nonzero(np.asarray(flag) != 0)[0]
    return idx[:cap].astype(np.uint32), int(idx.size)


def abft_capture(flag, flag_col, A_bits, W_bits, C_bits, cap_rows: int, cap_cols: int) -> dict:
    """The replay context of C = A W^T: per flagged row i, A[i, :] and C[i, :]; per flagged column
    j, W[j, :] (B's column j, as W is stored) and C[:, j].  The first cap rows and columns in index
    order are kept; the counts are of everything flagged."""
    ri, nr = capture_index(flag, cap_rows)
    out = {"row_idx": ri, "row_A": A_bits[ri], "row_C": C_bits[ri], "n_rows": nr}
    if flag_col is not None:
        ci, nc = capture_index(flag_col, cap_cols)
        out.update({"col_idx": ci, "col_W": W_bits[ci], "col_C": C_bits[:, ci].T.copy(), "n_cols": nc})
    return out


def wgrad_capture(flag, flag_col, dY_bits, X_bits, dW_bits, cap_rows: int, cap_cols: int) -> dict:
    """The replay context of dW = dY^T X: per flagged row n of dW, dY[:, n] (A's row) and dW[n, :];
    per flagged column k, X[:, k] (B's column) and dW[:, k]."""
    ri, nr = capture_index(flag, cap_rows)
    ci, nc = capture_index(flag_col, cap_cols)
    return {"row_idx": ri, "row_dY": dY_bits[:, ri].T.copy(), "row_dW": dW_bits[ri], "n_rows": nr,
            "col_idx": ci, "col_X": X_bits[:, ci].T.copy(), "col_dW": dW_bits[:, ci].T.copy(), "n_cols": nc}


def output_consistent(C_bits: np.ndarray, exact: np.ndarray, mag: np.ndarray, K: int) -> np.ndarray:
    """Whether each saved bf16 output can come from a correct product: within the float32
    accumulation bound g (1 + g) mag + 2 K 2^-126 (g = K 2^-22, mag = sum_k |a| |b|) of the exact
    value, then rounded to bf16 (2^-8 of the value, or 2^-134 if subnormal).  A replay of a
    correct computation reproduces such values; an output outside it was computed wrongly."""
    g = K * 2.0 ** -22
    e = g * (1.0 + g) * np.asarray(mag, dtype=np.float64) + 2.0 * K * 2.0 ** -126
    got = bf16_to_f64(C_bits)
    with np.errstate(invalid="ignore"):
        return np.abs(got - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134


def abft_replay_rows(row_A_bits, W_bits, row_C_bits) -> np.ndarray:
    """Per captured row: how many of its saved outputs a correct product cannot give (0: the
    saved row is consistent with its inputs; a replay confirms a fault where this is > 0)."""
    K = W_bits.shape[1]
    A = bf16_to_f64(row_A_bits)
    W = bf16_to_f64(W_bits)
    ok = output_consistent(row_C_bits, A @ W.T, np.abs(A) @ np.abs(W).T, K)
    return (~ok).sum(axis=1)


def abft_replay_pairs(cap: dict) -> np.ndarray:
    """Per captured (row r, column c) pair of a forward product: whether the saved C[i_r, j_c] is
    inconsistent with the saved operands A[i_r, :] and W[j_c, :] (1) or not (0)."""
    A = bf16_to_f64(cap["row_A"])  # [rows, K]
    W = bf16_to_f64(cap["col_W"])  # [cols, K]
    K = A.shape[1]
    saved = cap["row_C"][:, cap["col_idx"]]  # [rows, cols]: C[i_r, j_c]
    ok = output_consistent(saved, A @ W.T, np.abs(A) @ np.abs(W).T, K)
    return (~ok).astype(np.uint8)


def wgrad_replay_pairs(cap: dict) -> np.ndarray:
    """Per captured (row r, column c) pair of a weight-gradient product: whether the saved
    dW[n_r, k_c] is inconsistent with the saved operands dY[:, n_r] and X[:, k_c] (1) or not (0)."""
    dY = bf16_to_f64(cap["row_dY"])  # [rows, T]
    X = bf16_to_f64(cap["col_X"])    # [cols, T]
    T = dY.shape[1]
    saved = cap["row_dW"][:, cap["col_idx"]]  # [rows, cols]: dW[n_r, k_c]
    ok = output_consistent(saved, dY @ X.T, np.abs(dY) @ np.abs(X).T, T)
    return (~ok).astype(np.uint8)


# --------------------------------------------------------------------------
# Attention invariant  ([AEGIS] method section 3: in the attention backward
# dV = P^T dO and every row of the softmax P sums to 1, so 1^T dV = 1^T dO;
# the column sums of dV come from its float32 accumulator)
# --------------------------------------------------------------------------
def attn_probs(Q_bits: np.ndarray, K_bits: np.ndarray, lse: np.ndarray, scale: float, causal: bool,
               key0: int = 0) -> np.ndarray:
    """P [L, n] of one head, rebuilt as the backward does: exp(scale Q K^T - lse) with
    the forward's log-sum-exp per query row; causal masks key j > query i to 0.  The
    rows of K_bits are keys key0, key0 + 1, ... (all L keys by default)."""
    S = bf16_to_f64(Q_bits) @ bf16_to_f64(K_bits).T
    P = np.exp(S * float(np.float32(scale)) - np.asarray(lse, dtype=np.float64)[:, None])
    if causal:
        P = np.tril(P, -key0)  # keeps P[i, jj] where key key0 + jj <= query i
    return P


def attn_dv(P: np.ndarray, dO_bits: np.ndarray) -> np.ndarray:
    """dV = P^T dO of one head, float64."""
    return P.T @ bf16_to_f64(dO_bits)


def attn_bound(abs_colsum_do: np.ndarray, L: int) -> np.ndarray:
    """Bound on |1^T dV - 1^T dO| per column for a backward that rounds P to bf16
    and accumulates dV in float32 over the L query rows.

    Each probability may be off by 2^-8 of itself (its bf16 rounding, 2^-9, plus up
    to 2^-9 for the recomputed scores, the exponential and the forward's float32
    log-sum-exp), so a row of P sums to 1 within 2^-8 (1 + 2^-7); each float32
    accumulation step may lose two units in the last place of its partial sum
    (g = L 2^-22).  The column sums of the check itself are taken as exact (the
    oracle's are float64); a check that carries them in less precision adds its
    own term on top."""
    g = L * 2.0 ** -22
    rho = 1.0 + 2.0 ** -7
    return (2.0 ** -8 * rho + g * (1.0 + g) * rho) * np.asarray(abs_colsum_do, dtype=np.float64) + 2.0 ** -100


def attn_invariant(colsum_dv: np.ndarray, dO_bits: np.ndarray, tol_scale: float = 1.0) -> dict:
    """The invariant of one head: residual[c] = colsum_dv[c] - sum_i dO[i, c], the bound,
    and the column flags (flagged unless |residual| <= tol_scale * bound; NaN flags)."""
    dO = bf16_to_f64(dO_bits)
    L = dO.shape[0]
    residual = np.asarray(colsum_dv, dtype=np.float64) - dO.sum(axis=0)
    bound = attn_bound(np.abs(dO).sum(axis=0), L)
    with np.errstate(invalid="ignore"):
        flag = ~(np.abs(residual) <= tol_scale * bound)
    return {"residual": residual, "bound": bound, "flag": flag.astype(np.uint8), "n_flagged": int(flag.sum())}
