"""Replica-integrity scan for one GB300 GPU: thin Python binding of libsdc.

The compute lives in the CUDA kernels of libsdc.so (see include/sdc.h for the
C ABI).  This module only marshals arguments: the ``sdc_*`` functions mirror
the C entry points one to one (integer device addresses, sizes, a stream
handle), and ``Plan`` / ``vote`` / ``grad_average_scan`` wrap them for
torch tensors.  There is no fallback: when the library has not been built
(``python -m silent_corruption_checksums_gb300.build``) every call raises
ImportError.

Method: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" (weight fingerprints, strict-majority vote, non-finite
gradient checks) and the review page "Safeguarding LLM Training at Scale ..."
(xorsum fingerprint of a recomputed result).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB_PATH, is_stale

__all__ = [
    "SdcError", "DTYPE_RAW", "DTYPE_F32", "DTYPE_BF16", "DTYPE_F16", "MAX_REPLICAS",
    "SUSPECT_AGREE", "SUSPECT_SEVERAL", "SUSPECT_NO_MAJORITY", "GRAD_STATS_DTYPE", "VOTE_SUMMARY_DTYPE",
    "sdc_plan_create", "sdc_plan_destroy", "sdc_workspace_size", "sdc_plan_info", "sdc_fingerprint",
    "sdc_xorsum", "sdc_xorsum_compare", "sdc_vote", "sdc_grad_scan", "sdc_grad_average_scan_workspace_size",
    "sdc_grad_average_scan", "sdc_grad_average_scan_noalloc", "NOALLOC_SCRATCH_BYTES", "sdc_status_string", "sdc_last_error", "Plan", "vote", "xorsum_compare",
    "grad_average_scan", "AdamWFingerprint", "AdamWHparams", "sdc_opt_state_create", "sdc_opt_state_destroy",
    "sdc_adamw_fingerprint", "ring_audit", "ring_result", "sdc_ring_audit", "RING_SUMMARY_DTYPE", "decode_stats", "decode_summary", "pages_verdict", "library_path",
]

DTYPE_RAW, DTYPE_F32, DTYPE_BF16, DTYPE_F16 = 0, 1, 2, 3
MAX_REPLICAS = 64
SUSPECT_AGREE, SUSPECT_SEVERAL, SUSPECT_NO_MAJORITY = -1, -2, -3

# Mirrors of the C structs (include/sdc.h).
DESC_DTYPE = np.dtype([("ptr", "<u8"), ("numel", "<u8"), ("elem_size", "<u4"), ("dtype", "<u4")])
GRAD_STATS_DTYPE = np.dtype([("n_nan", "<u8"), ("n_inf", "<u8"), ("n_big", "<u8"), ("n_elems", "<u8"),
                             ("sumsq_finite", "<f8"), ("norm", "<f8"), ("nonfinite_fp32", "<u4"),
                             ("reserved", "<u4")])
RING_SUMMARY_DTYPE = np.dtype([("n_pairs", "<u4"), ("n_culprits", "<u4"), ("n_ambiguous", "<u4"),
                               ("reserved", "<u4")])
VOTE_SUMMARY_DTYPE = np.dtype([("diverged", "<u4"), ("no_majority", "<u4"), ("suspect_mask", "<u8"),
                               ("n_differing", "<u4"), ("n_no_majority", "<u4")])
assert DESC_DTYPE.itemsize == 24 and GRAD_STATS_DTYPE.itemsize == 56 and VOTE_SUMMARY_DTYPE.itemsize == 24


class SdcError(RuntimeError):
    """A libsdc call returned a non-zero status."""

    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn}: {sdc_status_string(status)} ({status}): {detail}")
        self.status = status


class AdamWHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("max_grad_norm", ctypes.c_float), ("step", ctypes.c_uint32),
                ("clip", ctypes.c_uint32)]


class _PlanOpts(ctypes.Structure):
    _fields_ = [("chunk_bytes", ctypes.c_uint32), ("ctas_per_sm", ctypes.c_uint32),
                ("skip_pointer_checks", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsdc.so not found at {LIB_PATH}; build it with "
                          "`python -m silent_corruption_checksums_gb300.build` (needs nvcc)")
    if is_stale():
        raise ImportError(f"libsdc.so at {LIB_PATH} is older than its sources; rebuild it with "
                          "`python -m silent_corruption_checksums_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, u64, u32, sz = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_size_t
    sig = {
        "sdc_plan_create": ([vp, u32, u32, ctypes.POINTER(_PlanOpts), ctypes.POINTER(vp)], ctypes.c_int),
        "sdc_plan_destroy": ([vp], ctypes.c_int),
        "sdc_workspace_size": ([vp], sz),
        "sdc_plan_info": ([vp, ctypes.POINTER(u64), ctypes.POINTER(u32), ctypes.POINTER(u32)], ctypes.c_int),
        "sdc_fingerprint": ([vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_xorsum": ([vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_xorsum_compare": ([vp, vp, u32, vp, vp, vp], ctypes.c_int),
        "sdc_vote": ([vp, u32, u32, vp, vp, vp, vp], ctypes.c_int),
        "sdc_grad_scan": ([vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_grad_average_scan_workspace_size": ([u64, u32, u32], sz),
        "sdc_grad_average_scan": ([ctypes.POINTER(vp), u32, vp, u64, u32, vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_grad_average_scan_noalloc": ([ctypes.POINTER(vp), u32, vp, u64, u32, vp, vp, vp], ctypes.c_int),
        "sdc_ring_audit": ([vp, u32, u32, u32, vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "sdc_opt_state_create": ([vp, ctypes.POINTER(vp), u32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                  ctypes.POINTER(vp)], ctypes.c_int),
        "sdc_opt_state_destroy": ([vp], ctypes.c_int),
        "sdc_adamw_fingerprint": ([vp, vp, ctypes.POINTER(AdamWHparams), vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_abft_workspace_size": ([u32, u32, u32], sz),
        "sdc_abft_gemm": ([vp, vp, vp, u32, u32, u32, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_abft_verify": ([vp, vp, u32, u32, u32, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
                            ctypes.c_int),
        "sdc_abft_weight_sums_workspace_size": ([u32, u32], sz),
        "sdc_abft_weight_sums": ([vp, u32, u32, vp, vp, sz, vp], ctypes.c_int),
        "sdc_abft_gemm_checked_workspace_size": ([u32, u32, u32], sz),
        "sdc_abft_gemm_checked": ([vp, vp, vp, u32, u32, u32, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, sz, vp],
                                  ctypes.c_int),
        "sdc_abft_wgrad_workspace_size": ([u32, u32, u32], sz),
        "sdc_abft_gemm_wgrad": ([vp, vp, vp, u32, u32, u32, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_abft_verify_wgrad": ([vp, vp, u32, u32, u32, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                   vp], ctypes.c_int),
        "sdc_abft_capture": ([vp, vp, vp, u32, u32, u32, vp, vp, u32, vp, vp, vp, u32, vp, vp, vp, vp, vp],
                             ctypes.c_int),
        "sdc_abft_capture_wgrad": ([vp, vp, vp, u32, u32, u32, vp, vp, u32, vp, vp, vp, u32, vp, vp, vp, vp, vp],
                                   ctypes.c_int),
        "sdc_abft_replay_workspace_size": ([u32, u32, u32], sz),
        "sdc_abft_replay": ([vp, u32, u32, u32, vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_abft_replay_pairs_workspace_size": ([u32, u32, u32], sz),
        "sdc_abft_replay_pairs": ([u32, u32, u32, u32, u32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
                                  ctypes.c_int),
        "sdc_abft_replay_wgrad_workspace_size": ([u32, u32, u32], sz),
        "sdc_abft_replay_wgrad": ([u32, u32, u32, u32, u32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp],
                                  ctypes.c_int),
        "sdc_attn_workspace_size": ([u32, u32, u32], sz),
        "sdc_attn_dv_check": ([vp, vp, vp, vp, u32, u32, u32, ctypes.c_float, u32, ctypes.c_float, vp, vp, vp, vp,
                               vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_attn_dv_check_grouped": ([vp, vp, vp, vp, u32, u32, u32, u32, ctypes.c_float, u32, ctypes.c_float, vp, vp,
                                       vp, vp, vp, vp, vp, vp, vp, sz, vp], ctypes.c_int),
        "sdc_selftest_bounded_wait": ([u32, vp, vp], ctypes.c_int),
        "sdc_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "sdc_last_error": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


class _Missing:
    """Stands in for the library until it is built: each use retries the load
    (the build step may have produced it since import) and raises if it is
    still missing."""

    def __init__(self, err: Exception):
        self.err = err

    def __getattr__(self, name):
        global _lib
        try:
            _lib = _load()
        except ImportError as e:
            raise ImportError(str(e)) from None
        return getattr(_lib, name)


try:
    _lib = _load()
except ImportError as _err:  # the build module must stay importable to create the library
    _lib = _Missing(_err)


def library_path() -> str:
    return LIB_PATH


def sdc_status_string(status: int) -> str:
    return _lib.sdc_status_string(status).decode()


def sdc_last_error() -> str:
    return _lib.sdc_last_error().decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise SdcError(fn, status, sdc_last_error())


# ---------------------------------------------------------------- C-ABI mirrors
def sdc_plan_create(descs: np.ndarray, T: int, R: int, chunk_bytes: int = 0, ctas_per_sm: int = 0,
                    skip_pointer_checks: bool = False) -> int:
    """descs: numpy array of DESC_DTYPE (R*T entries, replica-major). Returns the plan handle."""
    descs = np.ascontiguousarray(descs, dtype=DESC_DTYPE)
    opts = _PlanOpts(chunk_bytes, ctas_per_sm, 1 if skip_pointer_checks else 0, 0)
    out = ctypes.c_void_p()
    _check("sdc_plan_create", _lib.sdc_plan_create(descs.ctypes.data if descs.size else None, T, R,
                                                   ctypes.byref(opts), ctypes.byref(out)))
    return out.value


def sdc_plan_destroy(plan: int) -> None:
    _check("sdc_plan_destroy", _lib.sdc_plan_destroy(plan))


def sdc_workspace_size(plan: int) -> int:
    return int(_lib.sdc_workspace_size(plan))


def sdc_plan_info(plan: int) -> tuple[int, int, int]:
    n, g, b = ctypes.c_uint64(), ctypes.c_uint32(), ctypes.c_uint32()
    _check("sdc_plan_info", _lib.sdc_plan_info(plan, ctypes.byref(n), ctypes.byref(g), ctypes.byref(b)))
    return n.value, g.value, b.value


def sdc_fingerprint(plan: int, d_out: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_fingerprint", _lib.sdc_fingerprint(plan, d_out, d_ws, ws_bytes, stream))


def sdc_xorsum(plan: int, d_out: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_xorsum", _lib.sdc_xorsum(plan, d_out, d_ws, ws_bytes, stream))


def sdc_xorsum_compare(d_a: int, d_b: int, n: int, d_mismatch: int, d_diff: int, stream: int) -> None:
    _check("sdc_xorsum_compare", _lib.sdc_xorsum_compare(d_a, d_b, n, d_mismatch, d_diff, stream))


def sdc_vote(d_fp: int, R: int, T: int, d_suspect: int, d_mask: int, d_summary: int, stream: int) -> None:
    _check("sdc_vote", _lib.sdc_vote(d_fp, R, T, d_suspect, d_mask, d_summary, stream))


def sdc_grad_scan(plan: int, d_stats: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_grad_scan", _lib.sdc_grad_scan(plan, d_stats, d_ws, ws_bytes, stream))


def sdc_grad_average_scan_workspace_size(numel: int, n_bufs: int, dtype: int) -> int:
    return int(_lib.sdc_grad_average_scan_workspace_size(numel, n_bufs, dtype))


def sdc_grad_average_scan(bufs: list[int], d_avg: int, numel: int, dtype: int, d_pre: int, d_post: int,
                          d_ws: int, ws_bytes: int, stream: int) -> None:
    arr = (ctypes.c_void_p * max(1, len(bufs)))(*bufs)
    _check("sdc_grad_average_scan", _lib.sdc_grad_average_scan(arr, len(bufs), d_avg, numel, dtype, d_pre,
                                                               d_post, d_ws, ws_bytes, stream))


def sdc_ring_audit(d_table: int, n: int, L: int, offset: int, d_mismatch: int, d_hits: int, d_culprit: int,
                   d_ambiguous: int, d_summary: int, stream: int) -> None:
    _check("sdc_ring_audit", _lib.sdc_ring_audit(d_table, n, L, offset, d_mismatch, d_hits, d_culprit, d_ambiguous,
                                                 d_summary, stream))


def sdc_opt_state_create(plan: int, grads: list[int], grad_dtype: int, exp_avg: list[int],
                         exp_avg_sq: list[int]) -> int:
    arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(*xs)
    out = ctypes.c_void_p()
    _check("sdc_opt_state_create", _lib.sdc_opt_state_create(plan, arr(grads), grad_dtype, arr(exp_avg),
                                                             arr(exp_avg_sq), ctypes.byref(out)))
    return out.value


def sdc_opt_state_destroy(state: int) -> None:
    _check("sdc_opt_state_destroy", _lib.sdc_opt_state_destroy(state))


def sdc_adamw_fingerprint(plan: int, state: int, hp: AdamWHparams, d_post: int, d_fp_out: int, d_ws: int,
                          ws_bytes: int, stream: int) -> None:
    _check("sdc_adamw_fingerprint", _lib.sdc_adamw_fingerprint(plan, state, ctypes.byref(hp), d_post, d_fp_out, d_ws,
                                                               ws_bytes, stream))


NOALLOC_SCRATCH_BYTES = 16 << 20


def sdc_grad_average_scan_noalloc(bufs: list[int], d_avg: int, numel: int, dtype: int, d_pre: int, d_post: int,
                                  stream: int) -> None:
    """The average-scan on the library's fixed device scratch (no workspace, no allocation)."""
    arr = (ctypes.c_void_p * max(1, len(bufs)))(*bufs)
    _check("sdc_grad_average_scan_noalloc", _lib.sdc_grad_average_scan_noalloc(arr, len(bufs), d_avg, numel, dtype,
                                                                               d_pre, d_post, stream))


def sdc_abft_workspace_size(M: int, N: int, K: int) -> int:
    return int(_lib.sdc_abft_workspace_size(M, N, K))


def sdc_abft_gemm(d_A: int, d_W: int, d_C: int, M: int, N: int, K: int, d_rowsum: int, d_colsum: int,
                  d_aborted: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_gemm", _lib.sdc_abft_gemm(d_A, d_W, d_C, M, N, K, d_rowsum, d_colsum or None, d_aborted, d_ws,
                                               ws_bytes, stream))


def sdc_abft_weight_sums_workspace_size(N: int, K: int) -> int:
    return int(_lib.sdc_abft_weight_sums_workspace_size(N, K))


def sdc_abft_weight_sums(d_W: int, N: int, K: int, d_wsums: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_weight_sums", _lib.sdc_abft_weight_sums(d_W, N, K, d_wsums, d_ws, ws_bytes, stream))


def sdc_abft_gemm_checked_workspace_size(M: int, N: int, K: int) -> int:
    return int(_lib.sdc_abft_gemm_checked_workspace_size(M, N, K))


def sdc_abft_gemm_checked(d_A: int, d_W: int, d_C: int, M: int, N: int, K: int, d_wsums: int, tol_scale: float,
                          d_rowsum: int, d_residual: int, d_bound: int, d_flag: int, d_summary: int, d_aborted: int,
                          d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_gemm_checked",
           _lib.sdc_abft_gemm_checked(d_A, d_W, d_C, M, N, K, d_wsums, tol_scale, d_rowsum, d_residual, d_bound,
                                      d_flag, d_summary, d_aborted, d_ws, ws_bytes, stream))


def sdc_abft_wgrad_workspace_size(T: int, N: int, K: int) -> int:
    return int(_lib.sdc_abft_wgrad_workspace_size(T, N, K))


def sdc_abft_gemm_wgrad(d_dY: int, d_X: int, d_dW: int, T: int, N: int, K: int, d_rowsum: int, d_colsum: int,
                        d_aborted: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_gemm_wgrad", _lib.sdc_abft_gemm_wgrad(d_dY, d_X, d_dW, T, N, K, d_rowsum, d_colsum or None,
                                                           d_aborted, d_ws, ws_bytes, stream))


def sdc_abft_verify_wgrad(d_dY: int, d_X: int, T: int, N: int, K: int, d_rowsum: int, d_colsum: int,
                          tol_scale: float, d_residual: int, d_bound: int, d_flag: int, d_residual_col: int,
                          d_bound_col: int, d_flag_col: int, d_summary: int, d_ws: int, ws_bytes: int,
                          stream: int) -> None:
    _check("sdc_abft_verify_wgrad", _lib.sdc_abft_verify_wgrad(d_dY, d_X, T, N, K, d_rowsum, d_colsum or None,
                                                               tol_scale, d_residual, d_bound, d_flag,
                                                               d_residual_col or None, d_bound_col or None,
                                                               d_flag_col or None, d_summary, d_ws, ws_bytes, stream))


def sdc_abft_capture(d_A: int, d_W: int, d_C: int, M: int, N: int, K: int, d_flag: int, d_flag_col: int,
                     cap_rows: int, d_row_idx: int, d_row_A: int, d_row_C: int, cap_cols: int, d_col_idx: int,
                     d_col_W: int, d_col_C: int, d_counts: int, stream: int) -> None:
    _check("sdc_abft_capture", _lib.sdc_abft_capture(d_A, d_W, d_C, M, N, K, d_flag, d_flag_col or None, cap_rows,
                                                     d_row_idx or None, d_row_A or None, d_row_C or None, cap_cols,
                                                     d_col_idx or None, d_col_W or None, d_col_C or None, d_counts,
                                                     stream))


def sdc_abft_capture_wgrad(d_dY: int, d_X: int, d_dW: int, T: int, N: int, K: int, d_flag: int, d_flag_col: int,
                           cap_rows: int, d_row_idx: int, d_row_dY: int, d_row_dW: int, cap_cols: int,
                           d_col_idx: int, d_col_X: int, d_col_dW: int, d_counts: int, stream: int) -> None:
    _check("sdc_abft_capture_wgrad",
           _lib.sdc_abft_capture_wgrad(d_dY, d_X, d_dW, T, N, K, d_flag, d_flag_col or None, cap_rows,
                                       d_row_idx or None, d_row_dY or None, d_row_dW or None, cap_cols,
                                       d_col_idx or None, d_col_X or None, d_col_dW or None, d_counts, stream))


def sdc_abft_replay_workspace_size(cap_rows: int, N: int, K: int) -> int:
    return int(_lib.sdc_abft_replay_workspace_size(cap_rows, N, K))


def sdc_abft_replay(d_W: int, N: int, K: int, cap_rows: int, d_row_idx: int, d_row_A: int, d_row_C: int,
                    d_counts: int, d_ndiff: int, d_summary: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_replay", _lib.sdc_abft_replay(d_W, N, K, cap_rows, d_row_idx, d_row_A, d_row_C, d_counts,
                                                   d_ndiff, d_summary, d_ws, ws_bytes, stream))


def sdc_abft_replay_pairs_workspace_size(K: int, cap_rows: int, cap_cols: int) -> int:
    return int(_lib.sdc_abft_replay_pairs_workspace_size(K, cap_rows, cap_cols))


def sdc_abft_replay_pairs(M: int, N: int, K: int, cap_rows: int, cap_cols: int, d_row_idx: int, d_row_A: int,
                          d_row_C: int, d_col_idx: int, d_col_W: int, d_col_C: int, d_counts: int, d_differs: int,
                          d_summary: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_replay_pairs",
           _lib.sdc_abft_replay_pairs(M, N, K, cap_rows, cap_cols, d_row_idx, d_row_A, d_row_C, d_col_idx, d_col_W,
                                      d_col_C, d_counts, d_differs, d_summary, d_ws, ws_bytes, stream))


def sdc_abft_replay_wgrad_workspace_size(T: int, cap_rows: int, cap_cols: int) -> int:
    return int(_lib.sdc_abft_replay_wgrad_workspace_size(T, cap_rows, cap_cols))


def sdc_abft_replay_wgrad(T: int, N: int, K: int, cap_rows: int, cap_cols: int, d_row_idx: int, d_row_dY: int,
                          d_row_dW: int, d_col_idx: int, d_col_X: int, d_col_dW: int, d_counts: int, d_differs: int,
                          d_summary: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_replay_wgrad",
           _lib.sdc_abft_replay_wgrad(T, N, K, cap_rows, cap_cols, d_row_idx, d_row_dY, d_row_dW, d_col_idx, d_col_X,
                                      d_col_dW, d_counts, d_differs, d_summary, d_ws, ws_bytes, stream))


def sdc_abft_verify(d_A: int, d_W: int, M: int, N: int, K: int, d_rowsum: int, d_colsum: int, tol_scale: float,
                    d_residual: int, d_bound: int, d_flag: int, d_residual_col: int, d_bound_col: int,
                    d_flag_col: int, d_summary: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_abft_verify", _lib.sdc_abft_verify(d_A, d_W, M, N, K, d_rowsum, d_colsum or None, tol_scale,
                                                   d_residual, d_bound, d_flag, d_residual_col or None,
                                                   d_bound_col or None, d_flag_col or None, d_summary, d_ws,
                                                   ws_bytes, stream))


def sdc_attn_workspace_size(BH: int, L: int, D: int) -> int:
    return int(_lib.sdc_attn_workspace_size(BH, L, D))


def sdc_attn_dv_check(d_Q: int, d_K: int, d_dO: int, d_lse: int, BH: int, L: int, D: int, scale: float, causal: int,
                      tol_scale: float, d_dV: int, d_colsum_dv: int, d_colsum_do: int, d_residual: int, d_bound: int,
                      d_flag: int, d_summary: int, d_aborted: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_attn_dv_check", _lib.sdc_attn_dv_check(d_Q, d_K, d_dO, d_lse, BH, L, D, scale, causal, tol_scale,
                                                       d_dV, d_colsum_dv, d_colsum_do, d_residual, d_bound, d_flag,
                                                       d_summary, d_aborted, d_ws, ws_bytes, stream))


def sdc_attn_dv_check_grouped(d_Q: int, d_K: int, d_dO: int, d_lse: int, BH: int, group: int, L: int, D: int,
                              scale: float, causal: int, tol_scale: float, d_dV: int, d_colsum_dv: int,
                              d_colsum_do: int, d_residual: int, d_bound: int, d_flag: int, d_summary: int,
                              d_aborted: int, d_ws: int, ws_bytes: int, stream: int) -> None:
    _check("sdc_attn_dv_check_grouped",
           _lib.sdc_attn_dv_check_grouped(d_Q, d_K, d_dO, d_lse, BH, group, L, D, scale, causal, tol_scale, d_dV,
                                          d_colsum_dv, d_colsum_do, d_residual, d_bound, d_flag, d_summary, d_aborted,
                                          d_ws, ws_bytes, stream))


def sdc_selftest_bounded_wait(polls: int, d_status: int, stream: int) -> None:
    _check("sdc_selftest_bounded_wait", _lib.sdc_selftest_bounded_wait(polls, d_status, stream))


# ---------------------------------------------------------------- torch conveniences
def _torch():
    import torch
    return torch


def dtype_code(t) -> int:
    torch = _torch()
    return {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16, torch.float16: DTYPE_F16}.get(t.dtype, DTYPE_RAW)


def _stream_handle(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ws(nbytes: int, device):
    torch = _torch()
    if nbytes == 0:
        return None
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


class Plan:
    """A plan over R replicas x T tensors held as torch CUDA tensors.

    ``replicas[r][k]`` is replica r's copy of tensor k; tensors must be
    contiguous and stay allocated while the plan is used.  The plan's device
    tables and a workspace (from torch's allocator) are created once.
    """

    def __init__(self, replicas, chunk_bytes: int = 0, ctas_per_sm: int = 0, skip_pointer_checks: bool = False,
                 dtypes: list[int] | None = None):
        torch = _torch()
        self.R = len(replicas)
        self.T = len(replicas[0]) if self.R else 0
        descs = np.zeros(self.R * self.T, dtype=DESC_DTYPE)
        dev = None
        for r, ts in enumerate(replicas):
            if len(ts) != self.T:
                raise ValueError("every replica needs the same number of tensors")
            for k, t in enumerate(ts):
                if not t.is_contiguous():
                    raise ValueError("tensors must be contiguous")
                if t.numel() and not t.is_cuda:
                    raise ValueError("tensors must be CUDA tensors")
                dev = t.device if t.is_cuda else dev
                i = r * self.T + k
                descs[i] = (t.data_ptr() if t.numel() else 0, t.numel(), t.element_size(),
                            dtypes[k] if dtypes is not None else dtype_code(t))
        self.device = dev if dev is not None else torch.device("cuda", torch.cuda.current_device())
        self._keep = replicas
        with torch.cuda.device(self.device):
            self.handle = sdc_plan_create(descs, self.T, self.R, chunk_bytes, ctas_per_sm, skip_pointer_checks)
            self.ws_bytes = sdc_workspace_size(self.handle)
            self.ws = _ws(self.ws_bytes, self.device)
        self.n_chunks, self.grid, self.block = sdc_plan_info(self.handle)

    @classmethod
    def from_descs(cls, descs: np.ndarray, T: int, R: int, device, keep=None, **kw) -> "Plan":
        """Plan over raw descriptors (device addresses); ``keep`` holds the owning tensors."""
        self = cls.__new__(cls)
        self.R, self.T = R, T
        self.device = device
        self._keep = keep
        torch = _torch()
        with torch.cuda.device(device):
            self.handle = sdc_plan_create(descs, T, R, **kw)
            self.ws_bytes = sdc_workspace_size(self.handle)
            self.ws = _ws(self.ws_bytes, device)
        self.n_chunks, self.grid, self.block = sdc_plan_info(self.handle)
        return self

    def _ws_ptr(self) -> int:
        return self.ws.data_ptr() if self.ws is not None else 0

    def fingerprint(self, out=None, stream=None):
        """(S, W) per replica and tensor: int64 tensor [R, T, 2] holding the uint64 bits."""
        torch = _torch()
        if out is None:
            out = torch.empty((self.R, self.T, 2), dtype=torch.int64, device=self.device)
        sdc_fingerprint(self.handle, out.data_ptr(), self._ws_ptr(), self.ws_bytes, _stream_handle(stream))
        return out

    def xorsum(self, out=None, stream=None):
        """Xorsum per replica and tensor: int64 tensor [R, T] holding the uint64 bits."""
        torch = _torch()
        if out is None:
            out = torch.empty((self.R, self.T), dtype=torch.int64, device=self.device)
        sdc_xorsum(self.handle, out.data_ptr(), self._ws_ptr(), self.ws_bytes, _stream_handle(stream))
        return out

    def grad_scan(self, out=None, stream=None):
        """Gradient statistics per replica: uint8 tensor [R, 56] (decode with decode_stats)."""
        torch = _torch()
        if out is None:
            out = torch.empty((self.R, GRAD_STATS_DTYPE.itemsize), dtype=torch.uint8, device=self.device)
        sdc_grad_scan(self.handle, out.data_ptr(), self._ws_ptr(), self.ws_bytes, _stream_handle(stream))
        return out

    def close(self) -> None:
        if getattr(self, "handle", None):
            sdc_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class AdamWFingerprint:
    """Clip + AdamW step + fingerprint of the written weights for a Plan of F32 weights.

    ``grads``: T tensors (the averaged gradient, shared by the replicas);
    ``exp_avg``/``exp_avg_sq``: R x T float32 tensors.
    """

    def __init__(self, plan: "Plan", grads, exp_avg, exp_avg_sq):
        self.plan = plan
        self._keep = (grads, exp_avg, exp_avg_sq)
        gd = dtype_code(grads[0]) if grads else DTYPE_F32
        flat = lambda xss: [t.data_ptr() if t.numel() else 0 for ts in xss for t in ts]
        self.handle = sdc_opt_state_create(plan.handle, [g.data_ptr() if g.numel() else 0 for g in grads], gd,
                                           flat(exp_avg), flat(exp_avg_sq))

    def step(self, hp: dict, post=None, out=None, stream=None):
        torch = _torch()
        if out is None:
            out = torch.empty((self.plan.R, self.plan.T, 2), dtype=torch.int64, device=self.plan.device)
        h = AdamWHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"],
                         hp.get("max_grad_norm", 1.0), hp["step"], 1 if hp.get("clip") else 0)
        sdc_adamw_fingerprint(self.plan.handle, self.handle, h, post.data_ptr() if post is not None else 0,
                              out.data_ptr(), self.plan._ws_ptr(), self.plan.ws_bytes, _stream_handle(stream))
        return out

    def close(self):
        if getattr(self, "handle", None):
            sdc_opt_state_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def vote(fp, stream=None, out=None):
    """Strict-majority vote over an [R, T, 2] fingerprint tensor.

    Returns (suspect int32 [T], mask int64 [T], summary uint8 [24]).
    """
    torch = _torch()
    R, T = int(fp.shape[0]), int(fp.shape[1])
    if out is None:
        suspect = torch.empty(T, dtype=torch.int32, device=fp.device)
        mask = torch.empty(T, dtype=torch.int64, device=fp.device)
        summary = torch.empty(VOTE_SUMMARY_DTYPE.itemsize, dtype=torch.uint8, device=fp.device)
    else:
        suspect, mask, summary = out
    sdc_vote(fp.data_ptr(), R, T, suspect.data_ptr() if T else 0, mask.data_ptr() if T else 0,
             summary.data_ptr(), _stream_handle(stream))
    return suspect, mask, summary


def ring_audit(table, offset: int, stream=None):
    """Ring replay audit on an [n, 2, L] int64 table (row 0 own result, row 1 replay of the target).

    Returns (mismatch uint8 [n], hits int32 [n], culprit uint8 [n], ambiguous uint8 [n], summary uint8 [16]),
    mismatch/ambiguous indexed by the replayer r of pair ((r + offset) % n, r).
    """
    torch = _torch()
    n, L = int(table.shape[0]), int(table.shape[2])
    dev = table.device
    mism = torch.empty(n, dtype=torch.uint8, device=dev)
    hits = torch.empty(n, dtype=torch.int32, device=dev)
    cul = torch.empty(n, dtype=torch.uint8, device=dev)
    amb = torch.empty(n, dtype=torch.uint8, device=dev)
    summ = torch.empty(RING_SUMMARY_DTYPE.itemsize, dtype=torch.uint8, device=dev)
    z = lambda t: t.data_ptr() if n else 0
    sdc_ring_audit(table.data_ptr() if table.numel() else 0, n, L, offset, z(mism), z(hits), z(cul), z(amb),
                   summ.data_ptr(), _stream_handle(stream))
    return mism, hits, cul, amb, summ


def ring_result(mism, culprit, offset: int) -> dict:
    """Host view of a ring audit: the page's mismatched pairs (target, replayer), culprits, ambiguous pairs."""
    m = mism.cpu().tolist()
    n = len(m)
    c = culprit.cpu().tolist()
    pairs = [((r + offset) % n, r) for r in range(n) if m[r]]
    culprits = sorted(r for r in range(n) if c[r])
    ambiguous = [p for p in pairs if not (set(p) & set(culprits))]
    return {"pairs": pairs, "culprits": culprits, "ambiguous": ambiguous}


def xorsum_compare(a, b, stream=None):
    """Element-wise compare of two xorsum vectors: (mismatch uint8 [n], diff int64 [n])."""
    torch = _torch()
    n = int(a.numel())
    mism = torch.empty(n, dtype=torch.uint8, device=a.device)
    diff = torch.empty(n, dtype=torch.int64, device=a.device)
    sdc_xorsum_compare(a.data_ptr(), b.data_ptr(), n, mism.data_ptr() if n else 0, diff.data_ptr() if n else 0,
                       _stream_handle(stream))
    return mism, diff


def grad_average_scan(bufs, out=None, stream=None, ws=None):
    """Fused scan of the local gradients, their average, and the scan of the average.

    Returns (avg tensor, pre stats uint8 [n_bufs, 56], post stats uint8 [56]).
    """
    torch = _torch()
    numel = int(bufs[0].numel())
    code = dtype_code(bufs[0])
    dev = bufs[0].device
    if out is None:
        out = torch.empty_like(bufs[0])
    pre = torch.empty((len(bufs), GRAD_STATS_DTYPE.itemsize), dtype=torch.uint8, device=dev)
    post = torch.empty(GRAD_STATS_DTYPE.itemsize, dtype=torch.uint8, device=dev)
    need = sdc_grad_average_scan_workspace_size(numel, len(bufs), code)
    if ws is None or ws.numel() < need:
        ws = _ws(need, dev)
    sdc_grad_average_scan([b.data_ptr() for b in bufs], out.data_ptr(), numel, code, pre.data_ptr(),
                          post.data_ptr(), ws.data_ptr() if ws is not None else 0, need, _stream_handle(stream))
    return out, pre, post


class AbftGemm:
    """C = A . W^T on the tensor cores with the per-row accumulator checksum (and,
    with columns=True, the per-column one: the row + column configuration), and
    its check against A (W^T 1) (and (1^T A) W^T).  A: bf16 [M, K], W: bf16 [N, K],
    both contiguous CUDA tensors; M >= 1, N and K multiples of 8, K <= 2^20.  Output
    and scratch buffers are allocated once per shape and reused by every call."""

    def __init__(self, M: int, N: int, K: int, device, columns: bool = False):
        torch = _torch()
        self.M, self.N, self.K = M, N, K
        self.C = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.rowsum = torch.empty(M, dtype=torch.float64, device=device)
        self.aborted = torch.zeros(1, dtype=torch.int32, device=device)
        self.residual = torch.empty(M, dtype=torch.float64, device=device)
        self.bound = torch.empty(M, dtype=torch.float64, device=device)
        self.flag = torch.empty(M, dtype=torch.uint8, device=device)
        self.summary = torch.zeros(2, dtype=torch.int32, device=device)
        self.columns = columns
        if columns:
            self.colsum = torch.empty(N, dtype=torch.float64, device=device)
            self.residual_col = torch.empty(N, dtype=torch.float64, device=device)
            self.bound_col = torch.empty(N, dtype=torch.float64, device=device)
            self.flag_col = torch.empty(N, dtype=torch.uint8, device=device)
        self.ws_bytes = sdc_abft_workspace_size(M, N, K)
        self.ws = _ws(self.ws_bytes, device)

    def _ptr(self, name):
        return getattr(self, name).data_ptr() if self.columns else 0

    def _shape(self, A, W):
        if tuple(A.shape) != (self.M, self.K) or tuple(W.shape) != (self.N, self.K):
            raise ValueError(f"expected A [{self.M}, {self.K}] and W [{self.N}, {self.K}]")

    def gemm(self, A, W, stream=None):
        """The GEMM and its row checksums (self.C, self.rowsum; self.aborted != 0 if a wait gave up)."""
        self._shape(A, W)
        sdc_abft_gemm(A.data_ptr(), W.data_ptr(), self.C.data_ptr(), self.M, self.N, self.K, self.rowsum.data_ptr(),
                      self._ptr("colsum"), self.aborted.data_ptr(), self.ws.data_ptr(), self.ws_bytes,
                      _stream_handle(stream))
        return self.C

    def verify(self, A, W, tol_scale: float = 1.0, rowsum=None, stream=None):
        """The check (self.residual, self.bound, self.flag, self.summary[0] = flagged rows; with
        columns, self.residual_col, self.bound_col, self.flag_col, self.summary[1] = flagged columns)."""
        self._shape(A, W)
        rs = self.rowsum if rowsum is None else rowsum
        sdc_abft_verify(A.data_ptr(), W.data_ptr(), self.M, self.N, self.K, rs.data_ptr(), self._ptr("colsum"),
                        tol_scale, self.residual.data_ptr(), self.bound.data_ptr(), self.flag.data_ptr(),
                        self._ptr("residual_col"), self._ptr("bound_col"), self._ptr("flag_col"),
                        self.summary.data_ptr(), self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))
        return self.flag

    def __call__(self, A, W, tol_scale: float = 1.0, stream=None):
        self.gemm(A, W, stream)
        self.verify(A, W, tol_scale, stream=stream)
        return self.C

    def weight_sums(self, W, stream=None):
        """W's column sums for the fused check (self.wsums, float32 [K, 2]); valid until W changes."""
        torch = _torch()
        if tuple(W.shape) != (self.N, self.K):
            raise ValueError(f"expected W [{self.N}, {self.K}]")
        if not hasattr(self, "wsums"):
            self.wsums = torch.empty((self.K, 2), dtype=torch.float32, device=self.C.device)
            self._wsb = sdc_abft_weight_sums_workspace_size(self.N, self.K)
            self._wsws = _ws(self._wsb, self.C.device)
        sdc_abft_weight_sums(W.data_ptr(), self.N, self.K, self.wsums.data_ptr(), self._wsws.data_ptr(), self._wsb,
                             _stream_handle(stream))
        return self.wsums

    def gemm_checked(self, A, W, tol_scale: float = 1.0, stream=None):
        """The GEMM with its row check fused into it, against self.wsums (weight_sums(W) first):
        self.C, self.rowsum, self.residual, self.bound, self.flag, self.summary[0]."""
        self._shape(A, W)
        if not hasattr(self, "wsums"):
            raise ValueError("call weight_sums(W) first")
        if not hasattr(self, "_cws"):
            self._cwsb = sdc_abft_gemm_checked_workspace_size(self.M, self.N, self.K)
            self._cws = _ws(self._cwsb, self.C.device)
        sdc_abft_gemm_checked(A.data_ptr(), W.data_ptr(), self.C.data_ptr(), self.M, self.N, self.K,
                              self.wsums.data_ptr(), tol_scale, self.rowsum.data_ptr(), self.residual.data_ptr(),
                              self.bound.data_ptr(), self.flag.data_ptr(), self.summary.data_ptr(),
                              self.aborted.data_ptr(), self._cws.data_ptr(), self._cwsb, _stream_handle(stream))
        return self.C

    def capture(self, A, W, cap_rows: int = 8, cap_cols: int = 8, flag=None, flag_col=None, stream=None) -> dict:
        """The replay context of the flagged rows (and, with columns, columns) of the last product:
        {"row_idx", "row_A", "row_C", "col_idx", "col_W", "col_C", "counts"} as device tensors
        (counts: flagged rows and columns, also past the caps).  flag / flag_col select other
        rows or columns than the check's flags."""
        torch = _torch()
        self._shape(A, W)
        dev = self.C.device
        f = self.flag if flag is None else flag
        fc = (self.flag_col if self.columns else None) if flag_col is None else flag_col
        out = {"row_idx": torch.zeros(cap_rows, dtype=torch.int32, device=dev),
               "row_A": torch.zeros((cap_rows, self.K), dtype=torch.bfloat16, device=dev),
               "row_C": torch.zeros((cap_rows, self.N), dtype=torch.bfloat16, device=dev),
               "col_idx": torch.zeros(cap_cols, dtype=torch.int32, device=dev),
               "col_W": torch.zeros((cap_cols, self.K), dtype=torch.bfloat16, device=dev),
               "col_C": torch.zeros((cap_cols, self.M), dtype=torch.bfloat16, device=dev),
               "counts": torch.zeros(2, dtype=torch.int32, device=dev), "cap_rows": cap_rows,
               "cap_cols": cap_cols}
        c = cap_cols if fc is not None else 0
        sdc_abft_capture(A.data_ptr(), W.data_ptr(), self.C.data_ptr(), self.M, self.N, self.K, f.data_ptr(),
                         fc.data_ptr() if fc is not None else 0, cap_rows, out["row_idx"].data_ptr(),
                         out["row_A"].data_ptr(), out["row_C"].data_ptr(), c, out["col_idx"].data_ptr() if c else 0,
                         out["col_W"].data_ptr() if c else 0, out["col_C"].data_ptr() if c else 0,
                         out["counts"].data_ptr(), _stream_handle(stream))
        return out

    def replay(self, W, cap: dict, stream=None):
        """Recompute the captured rows against W with the same tensor-core kernel: (ndiff [cap_rows],
        summary [2]) as device tensors -- per row the outputs not reproduced bit for bit; summary:
        rows with any, and the replay GEMM's abort flag."""
        torch = _torch()
        n = cap["cap_rows"]
        dev = W.device
        ndiff = torch.zeros(n, dtype=torch.int32, device=dev)
        summary = torch.zeros(2, dtype=torch.int32, device=dev)
        wsb = sdc_abft_replay_workspace_size(n, self.N, self.K)
        ws = _ws(wsb, dev)
        sdc_abft_replay(W.data_ptr(), self.N, self.K, n, cap["row_idx"].data_ptr(), cap["row_A"].data_ptr(),
                        cap["row_C"].data_ptr(), cap["counts"].data_ptr(), ndiff.data_ptr(), summary.data_ptr(),
                        ws.data_ptr(), wsb, _stream_handle(stream))
        return ndiff, summary

    def replay_pairs(self, cap: dict, stream=None):
        """Recompute every captured (row, column) output from the captured A row and W row alone (the
        row + column configuration): (differs [cap_rows, cap_cols] uint8, summary [2]) as device tensors."""
        torch = _torch()
        nr, nc = cap["cap_rows"], cap["cap_cols"]
        dev = self.C.device
        differs = torch.zeros((nr, nc), dtype=torch.uint8, device=dev)
        summary = torch.zeros(2, dtype=torch.int32, device=dev)
        wsb = sdc_abft_replay_pairs_workspace_size(self.K, nr, nc)
        ws = _ws(wsb, dev)
        sdc_abft_replay_pairs(self.M, self.N, self.K, nr, nc, cap["row_idx"].data_ptr(), cap["row_A"].data_ptr(),
                              cap["row_C"].data_ptr(), cap["col_idx"].data_ptr(), cap["col_W"].data_ptr(),
                              cap["col_C"].data_ptr(), cap["counts"].data_ptr(), differs.data_ptr(),
                              summary.data_ptr(), ws.data_ptr(), wsb, _stream_handle(stream))
        return differs, summary


class AbftWgrad:
    """dW = dY^T . X (a linear layer's weight gradient) on the tensor cores with the
    accumulator's row checksums and, with columns=True (the default: the page's
    row + column configuration, which covers wgrad), column checksums, and their
    check against dY^T (X 1) and (dY 1)^T X.  dY: bf16 [T, N], X: bf16 [T, K], both
    token-major contiguous CUDA tensors; T >= 1, N and K multiples of 8.  Outputs
    and scratch are allocated once per shape and reused by every call."""

    def __init__(self, T: int, N: int, K: int, device, columns: bool = True):
        torch = _torch()
        self.T, self.N, self.K = T, N, K
        self.dW = torch.empty((N, K), dtype=torch.bfloat16, device=device)
        f64 = dict(dtype=torch.float64, device=device)
        self.rowsum, self.residual, self.bound = (torch.empty(N, **f64) for _ in range(3))
        self.flag = torch.empty(N, dtype=torch.uint8, device=device)
        self.aborted = torch.zeros(1, dtype=torch.int32, device=device)
        self.summary = torch.zeros(2, dtype=torch.int32, device=device)
        self.columns = columns
        if columns:
            self.colsum, self.residual_col, self.bound_col = (torch.empty(K, **f64) for _ in range(3))
            self.flag_col = torch.empty(K, dtype=torch.uint8, device=device)
        self.ws_bytes = sdc_abft_wgrad_workspace_size(T, N, K)
        self.ws = _ws(self.ws_bytes, device)

    def _ptr(self, name):
        return getattr(self, name).data_ptr() if self.columns else 0

    def _shape(self, dY, X):
        if tuple(dY.shape) != (self.T, self.N) or tuple(X.shape) != (self.T, self.K):
            raise ValueError(f"expected dY [{self.T}, {self.N}] and X [{self.T}, {self.K}]")

    def gemm(self, dY, X, stream=None):
        """dW and its checksums (self.dW, self.rowsum, self.colsum; self.aborted != 0 if a wait gave up)."""
        self._shape(dY, X)
        sdc_abft_gemm_wgrad(dY.data_ptr(), X.data_ptr(), self.dW.data_ptr(), self.T, self.N, self.K,
                            self.rowsum.data_ptr(), self._ptr("colsum"), self.aborted.data_ptr(), self.ws.data_ptr(),
                            self.ws_bytes, _stream_handle(stream))
        return self.dW

    def verify(self, dY, X, tol_scale: float = 1.0, stream=None):
        """The check (self.residual, self.bound, self.flag, self.summary[0] = flagged rows; with
        columns, self.residual_col, self.bound_col, self.flag_col, self.summary[1])."""
        self._shape(dY, X)
        sdc_abft_verify_wgrad(dY.data_ptr(), X.data_ptr(), self.T, self.N, self.K, self.rowsum.data_ptr(),
                              self._ptr("colsum"), tol_scale, self.residual.data_ptr(), self.bound.data_ptr(),
                              self.flag.data_ptr(), self._ptr("residual_col"), self._ptr("bound_col"),
                              self._ptr("flag_col"), self.summary.data_ptr(), self.ws.data_ptr(), self.ws_bytes,
                              _stream_handle(stream))
        return self.flag

    def __call__(self, dY, X, tol_scale: float = 1.0, stream=None):
        self.gemm(dY, X, stream)
        self.verify(dY, X, tol_scale, stream=stream)
        return self.dW

    def capture(self, dY, X, cap_rows: int = 8, cap_cols: int = 8, flag=None, flag_col=None, stream=None) -> dict:
        """The replay context of the flagged rows and columns of the last dW: {"row_idx", "row_dY"
        (dY's columns), "row_dW", "col_idx", "col_X" (X's columns), "col_dW", "counts"}."""
        torch = _torch()
        self._shape(dY, X)
        dev = self.dW.device
        f = self.flag if flag is None else flag
        fc = (self.flag_col if self.columns else None) if flag_col is None else flag_col
        out = {"row_idx": torch.zeros(cap_rows, dtype=torch.int32, device=dev),
               "row_dY": torch.zeros((cap_rows, self.T), dtype=torch.bfloat16, device=dev),
               "row_dW": torch.zeros((cap_rows, self.K), dtype=torch.bfloat16, device=dev),
               "col_idx": torch.zeros(cap_cols, dtype=torch.int32, device=dev),
               "col_X": torch.zeros((cap_cols, self.T), dtype=torch.bfloat16, device=dev),
               "col_dW": torch.zeros((cap_cols, self.N), dtype=torch.bfloat16, device=dev),
               "counts": torch.zeros(2, dtype=torch.int32, device=dev), "cap_rows": cap_rows,
               "cap_cols": cap_cols}
        c = cap_cols if fc is not None else 0
        sdc_abft_capture_wgrad(dY.data_ptr(), X.data_ptr(), self.dW.data_ptr(), self.T, self.N, self.K, f.data_ptr(),
                               fc.data_ptr() if fc is not None else 0, cap_rows, out["row_idx"].data_ptr(),
                               out["row_dY"].data_ptr(), out["row_dW"].data_ptr(), c,
                               out["col_idx"].data_ptr() if c else 0, out["col_X"].data_ptr() if c else 0,
                               out["col_dW"].data_ptr() if c else 0, out["counts"].data_ptr(), _stream_handle(stream))
        return out

    def replay(self, cap: dict, stream=None):
        """Recompute every captured (row, column) output from the captured dY and X columns alone:
        (differs [cap_rows, cap_cols] uint8, summary [2]) as device tensors."""
        torch = _torch()
        nr, nc = cap["cap_rows"], cap["cap_cols"]
        dev = self.dW.device
        differs = torch.zeros((nr, nc), dtype=torch.uint8, device=dev)
        summary = torch.zeros(2, dtype=torch.int32, device=dev)
        wsb = sdc_abft_replay_wgrad_workspace_size(self.T, nr, nc)
        ws = _ws(wsb, dev)
        sdc_abft_replay_wgrad(self.T, self.N, self.K, nr, nc, cap["row_idx"].data_ptr(), cap["row_dY"].data_ptr(),
                              cap["row_dW"].data_ptr(), cap["col_idx"].data_ptr(), cap["col_X"].data_ptr(),
                              cap["col_dW"].data_ptr(), cap["counts"].data_ptr(), differs.data_ptr(),
                              summary.data_ptr(), ws.data_ptr(), wsb, _stream_handle(stream))
        return differs, summary


class AttnDvCheck:
    """The dV half of the attention backward with the invariant 1^T dV = 1^T dO.
    Q, dO: bf16 [BH, L, 128] contiguous CUDA tensors; lse: float32 [BH, L], the
    forward's log-sum-exp; K: bf16 [BH / group, L, 128] (group query heads per K/V
    head; 1: plain multi-head attention).  dV and the per-column results are per
    K/V head.  Outputs and scratch are allocated once per shape."""

    def __init__(self, BH: int, L: int, device, D: int = 128, group: int = 1):
        torch = _torch()
        if group < 1 or BH % group:
            raise ValueError("group must divide BH")
        self.BH, self.L, self.D, self.group = BH, L, D, group
        kv = BH // group
        self.dV = torch.empty((kv, L, D), dtype=torch.bfloat16, device=device)
        f64 = dict(dtype=torch.float64, device=device)
        self.colsum_dv = torch.empty((kv, D), **f64)
        self.colsum_do = torch.empty((kv, D), **f64)
        self.residual = torch.empty((kv, D), **f64)
        self.bound = torch.empty((kv, D), **f64)
        self.flag = torch.empty((kv, D), dtype=torch.uint8, device=device)
        self.summary = torch.zeros(2, dtype=torch.int32, device=device)
        self.aborted = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_bytes = sdc_attn_workspace_size(BH, L, D)
        self.ws = _ws(self.ws_bytes, device)

    def __call__(self, Q, K, dO, lse, scale: float, causal: bool, tol_scale: float = 1.0, stream=None):
        for t in (Q, dO):
            if tuple(t.shape) != (self.BH, self.L, self.D):
                raise ValueError(f"expected [{self.BH}, {self.L}, {self.D}] Q and dO")
        if tuple(K.shape) != (self.BH // self.group, self.L, self.D):
            raise ValueError(f"expected K [{self.BH // self.group}, {self.L}, {self.D}]")
        sdc_attn_dv_check_grouped(Q.data_ptr(), K.data_ptr(), dO.data_ptr(), lse.data_ptr(), self.BH, self.group,
                                  self.L, self.D, scale, int(bool(causal)), tol_scale, self.dV.data_ptr(),
                                  self.colsum_dv.data_ptr(), self.colsum_do.data_ptr(), self.residual.data_ptr(),
                                  self.bound.data_ptr(), self.flag.data_ptr(), self.summary.data_ptr(),
                                  self.aborted.data_ptr(), self.ws.data_ptr(), self.ws_bytes, _stream_handle(stream))
        return self.dV


# ---------------------------------------------------------------- host-side decoding
def decode_stats(raw) -> list[dict]:
    """Decode sdc_grad_stats records (bytes, numpy or a CPU/GPU uint8 tensor) into dicts."""
    if hasattr(raw, "cpu"):
        raw = raw.cpu().numpy()
    arr = np.frombuffer(np.ascontiguousarray(raw).tobytes(), dtype=GRAD_STATS_DTYPE)
    return [{k: (float(rec[k]) if k in ("sumsq_finite", "norm") else int(rec[k]))
             for k in GRAD_STATS_DTYPE.names if k != "reserved"} for rec in arr]


def decode_summary(raw) -> dict:
    if hasattr(raw, "cpu"):
        raw = raw.cpu().numpy()
    rec = np.frombuffer(np.ascontiguousarray(raw).tobytes(), dtype=VOTE_SUMMARY_DTYPE)[0]
    return {k: int(rec[k]) for k in VOTE_SUMMARY_DTYPE.names}


def pages_verdict(summary: dict) -> dict:
    """The page's result dict {"diverged", "suspects"} from a decoded summary."""
    if not summary["diverged"]:
        return {"diverged": False, "suspects": []}
    if summary["no_majority"]:
        return {"diverged": True, "suspects": None}
    m = summary["suspect_mask"]
    return {"diverged": True, "suspects": [r for r in range(MAX_REPLICAS) if (m >> r) & 1]}
