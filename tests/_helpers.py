"""Helpers shared by the tests: host copies of device tensors for the oracle,
and conversions of the library's outputs to Python ints."""
from __future__ import annotations

import numpy as np
import torch

M64 = (1 << 64) - 1
_NP_INT = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}
_T_INT = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits of a tensor as a host numpy array of the same item size."""
    es = t.element_size()
    flat = t.detach().reshape(-1)
    return flat.view(_T_INT[es]).cpu().numpy().view(_NP_INT[es])


def u64(x: int) -> int:
    return int(x) & M64


def fp_table(out: torch.Tensor) -> list[list[tuple[int, int]]]:
    """[R, T, 2] int64 device tensor -> nested lists of (S, W) as unsigned ints."""
    a = out.cpu().numpy().view(np.uint64)
    return [[(int(a[r, k, 0]), int(a[r, k, 1])) for k in range(a.shape[1])] for r in range(a.shape[0])]


def oracle_fp_table(replicas, threads: int = 1):
    import oracle
    return [[oracle.fingerprint(host_bits(t), threads=threads) for t in ts] for ts in replicas]


def rel_err(a: float, b: float) -> float:
    if a == b:
        return 0.0
    return abs(a - b) / max(abs(b), 1e-300)


def stats_match(gpu: dict, ref: dict, rtol: float = 1e-10) -> None:
    """Counts, flags and element totals exactly; sumsq and norm within rtol (norm class-wise)."""
    import math
    for k in ("n_nan", "n_inf", "n_big", "n_elems"):
        assert gpu[k] == ref[k], (k, gpu[k], ref[k])
    assert rel_err(gpu["sumsq_finite"], ref["sumsq_finite"]) <= rtol, (gpu["sumsq_finite"], ref["sumsq_finite"])
    if math.isnan(ref["norm"]):
        assert math.isnan(gpu["norm"])
    elif math.isinf(ref["norm"]):
        assert gpu["norm"] == ref["norm"]
    else:
        assert rel_err(gpu["norm"], ref["norm"]) <= rtol, (gpu["norm"], ref["norm"])
    # the float32 flag is exact unless the squared norm sits within rtol of FLT_MAX
    import oracle
    if abs(ref["sumsq_finite"] - oracle.FLT_MAX) > 1e-9 * oracle.FLT_MAX:
        assert gpu["nonfinite_fp32"] == ref["nonfinite_fp32"]


def verifier_own_slack(n_sum: int, K: int) -> float:
    """The GEMM check kernel's own term, relative to the magnitude: it sums in plain float32
    chains of at most 8 terms folded into float32 pairs (below 20 2^-24 of the magnitude in
    all) and carries the pairs and their merges at about 48 bits ((n_sum + K + 64) 2^-44).
    Its bound adds this term, and its residual agrees with exact sums to it."""
    return 20.0 * 2.0 ** -24 + (n_sum + K + 64) * 2.0 ** -44


def verifier_mag_slack(n_sum: int, K: int) -> float:
    """How far above the exact magnitude the GEMM check's raised magnitude may sit, relative:
    it sums |W| and |A| |W^T 1| in plain float32 chains (at most n_sum / 8 rows and K / 8 + 8
    columns long, at most K / 64 + 1 splits) and raises the result by twice their length in
    units of 2^-24, so that it is never below the exact magnitude."""
    return 2.0 * (n_sum / 8 + K / 4 + 32) * 2.0 ** -24


def assert_verifier_bound(kernel_bound, method_bound, mag, n_sum: int, K: int) -> None:
    """The kernel's bound is never below the method's (no clean output can flag for the
    kernel's own rounding), and above it by no more than the kernel's own terms: its own
    sums (verifier_own_slack) and its raised magnitude (verifier_mag_slack)."""
    import numpy as np
    kb, mb, mg = (np.asarray(x, dtype=np.float64) for x in (kernel_bound, method_bound, mag))
    assert np.all(kb >= mb * (1.0 - 1e-12)), float(np.min(kb / mb))
    top = (mb + verifier_own_slack(n_sum, K) * mg) * (1.0 + verifier_mag_slack(n_sum, K)) * (1.0 + 1e-12)
    assert np.all(kb <= top), float(np.max(kb / top))


def assert_wgrad_bound(kernel_bound, method_bound, mag, n_sum: int, T: int) -> None:
    """The weight-gradient check's bound against the method's: its own sums as the forward
    check's with the T tokens as the contraction, and its magnitude raised by at most
    2 (T / 8 + n_sum / 64 + 20) 2^-24 (a slab warp's rows, a row-sum lane's terms, merges)."""
    import numpy as np
    kb, mb, mg = (np.asarray(x, dtype=np.float64) for x in (kernel_bound, method_bound, mag))
    assert np.all(kb >= mb * (1.0 - 1e-12)), float(np.min(kb / mb))
    raise_ = 2.0 * (T / 8 + n_sum / 64 + 20) * 2.0 ** -24
    top = (mb + verifier_own_slack(n_sum, T) * mg) * (1.0 + raise_) * (1.0 + 1e-12)
    assert np.all(kb <= top), float(np.max(kb / top))


# The attention check's own terms, relative to A = sum_i |dO[i, c]|: its column sums are float32
# pairs (2^-40) of plain 8-row chains (below 8 2^-24 each, counted twice: 2^-20), and it raises A by
# 2^-21 so that its bound never falls below the method's whatever the chains lost.
ATTN_OWN_SLACK = 2.0 ** -40 + 2.0 ** -20
ATTN_MAG_RAISE = 2.0 ** -21


def assert_attn_bound(kernel_bound, method_bound, abs_colsum) -> None:
    """The attention check's bound is never below the method's and above it by at most its own
    terms (ATTN_OWN_SLACK of sum |dO|, and the raise of sum |dO|)."""
    import numpy as np
    kb, mb, a = (np.asarray(x, dtype=np.float64) for x in (kernel_bound, method_bound, abs_colsum))
    assert np.all(kb >= mb * (1.0 - 1e-12)), float(np.min(kb / mb))
    top = (mb + ATTN_OWN_SLACK * a) * (1.0 + 2.0 * ATTN_MAG_RAISE) * (1.0 + 1e-12)
    assert np.all(kb <= top), float(np.max(kb / top))
