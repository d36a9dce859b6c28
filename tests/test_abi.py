"""The C ABI library loads on a CPU-only host, exports every entry point the
header declares, and its host-side validation rejects bad arguments before
touching the GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdc.h")


@pytest.fixture(scope="module")
def sdc():
    from silent_corruption_checksums_gb300 import build
    build.build()
    import silent_corruption_checksums_gb300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdc_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(sdc):
    names = _declared_functions()
    assert len(names) >= 13
    lib = ctypes.CDLL(sdc.library_path())
    for n in names:
        assert hasattr(lib, n), n


def test_struct_layouts_match_header(sdc):
    assert sdc.DESC_DTYPE.itemsize == 24
    assert sdc.GRAD_STATS_DTYPE.itemsize == 56
    assert sdc.VOTE_SUMMARY_DTYPE.itemsize == 24


def test_status_strings(sdc):
    assert sdc.sdc_status_string(0) == "SDC_OK"
    assert sdc.sdc_status_string(5) == "SDC_ERR_WS_TOO_SMALL"
    assert sdc.sdc_status_string(99) == "SDC_ERR_UNKNOWN"


def _descs(entries):
    d = np.zeros(len(entries), dtype=np.dtype([("ptr", "<u8"), ("numel", "<u8"), ("elem_size", "<u4"),
                                               ("dtype", "<u4")]))
    for i, e in enumerate(entries):
        d[i] = e
    return d


def test_host_validation_without_gpu(sdc):
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([]), 0, 0)
    assert ei.value.status == 4  # R == 0
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4096, 10, 4, 1)] * 65), 1, 65)
    assert ei.value.status == 4  # R > 64
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4096, 10, 3, 0)]), 1, 1)
    assert ei.value.status == 2  # element size 3
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4096, 10, 2, 1)]), 1, 1)
    assert ei.value.status == 2  # f32 with 2-byte elements
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4096, 10, 4, 9)]), 1, 1)
    assert ei.value.status == 7  # unknown dtype
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4096, 10, 4, 1), (8192, 11, 4, 1)]), 1, 2)
    assert ei.value.status == 3  # replica 1 has another numel
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(0, 10, 4, 1)]), 1, 1)
    assert ei.value.status == 1  # NULL with elements
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4098, 10, 4, 1)]), 1, 1)
    assert ei.value.status == 8  # not aligned to the element size
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(_descs([(4096, 10, 4, 1)]), 1, 1, chunk_bytes=5000)
    assert ei.value.status == 9
    assert "chunk_bytes" in sdc.sdc_last_error()
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_vote(0, 0, 1, 0, 0, 0, 0)
    assert ei.value.status == 4
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_grad_average_scan([], 0, 10, 2, 0, 0, 0, 0, 0)
    assert ei.value.status == 4
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_grad_average_scan([4096], 8192, 10, 0, 8, 8, 0, 0, 0)
    assert ei.value.status == 7
    # per-task partials (one 16 KiB task x 5 streams x 24 B, rounded to 256) + 128 group sums per stream
    # (32 B each: the counts are 64-bit)
    assert sdc.sdc_grad_average_scan_workspace_size(0, 4, 2) == 5 * 128 * 32
    assert sdc.sdc_grad_average_scan_workspace_size(8192, 4, 2) == 256 + 5 * 128 * 32
    assert sdc.sdc_grad_average_scan_workspace_size(8192, 9, 2) == 0  # more than 8 buffers
    sdc.sdc_xorsum_compare(0, 0, 0, 0, 0, 0)  # n == 0 is a no-op
    # GEMM checksum: operands checked, then shapes, before any CUDA call
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm(0, 4096, 8192, 128, 256, 64, 0, 0, 0, 0, 0, 0)
    assert ei.value.status == 1
    for M, N, K in [(100, 260, 64), (128, 200, 60), (0, 256, 64), (128, 0, 64), (128, 256, 0),
                    (128, 256, (1 << 20) + 8), (128, 256, 1 << 21)]:
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_gemm(4096, 8192, 16384, M, N, K, 0, 0, 0, 0, 0, 0)
        assert ei.value.status == 9, (M, N, K)
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_verify(4096, 8192, M, N, K, 0, 0, 1.0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0)
        assert ei.value.status == 9, (M, N, K)
    # row partials (ceil(N/256) per row), column partials (ceil(M/128) per column), W's and A's column sums
    # (K x 8 bytes each: the sum and the magnitude in float32), slabs of K x 16 bytes for both column
    # sums (slabs = min(456 / ceil(K / 256), 64, rows / 8) each), both checks' split partials (16 bytes per
    # row and split; one split when K / 8 < 128), the last-block counters (a word per 32-row block of both
    # sides, or per 256 columns of both), the abort word; each rounded up to 256 bytes
    assert sdc.sdc_abft_workspace_size(128, 512, 64) == (2048 + 1 * 512 * 8 + 2 * 512 + (64 + 16) * 64 * 16
                                                         + (128 + 512) * 16 + 256 + 256)
    assert sdc.sdc_abft_workspace_size(1000, 256, 100) == (8192 + 8 * 256 * 8 + 2 * 1024 + (32 + 64) * 100 * 16
                                                           + 20224 + 256 + 256)
    # weight-gradient GEMM checksum: operands, then shapes (T tokens in 1..2^20, N and K multiples of 8)
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_gemm_wgrad(0, 4096, 8192, 128, 256, 64, 0, 0, 0, 0, 0, 0)
    assert ei.value.status == 1
    for T, N, K in [(0, 256, 64), (128, 0, 64), (128, 256, 0), (128, 260, 64), (128, 256, 60), ((1 << 20) + 1, 256, 64)]:
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_gemm_wgrad(4096, 8192, 16384, T, N, K, 0, 0, 0, 0, 0, 0)
        assert ei.value.status == 9, (T, N, K)
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_verify_wgrad(4096, 8192, T, N, K, 0, 0, 1.0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0)
        assert ei.value.status == 9, (T, N, K)
    # row partials (ceil(K/256) per dW row), column partials (ceil(N/128) per column), X's and dY's row
    # sums (8 bytes per token each), slabs of 16 bytes per column of each operand
    # (min(456 / ceil(n / 256), 64, T / 8) slabs each), the last-block counters (a word per 256 columns of
    # each), the abort word; each rounded up to 256 bytes
    assert sdc.sdc_abft_wgrad_workspace_size(512, 256, 128) == (2048 + 2048 + 4096 + 4096 + 64 * (256 + 128) * 16
                                                                + 256 + 256)
    assert sdc.sdc_abft_wgrad_workspace_size(100, 8, 1000) == (256 + 8192 + 1024 + 1024 + 12 * (8 + 1000) * 16
                                                               + 256 + 256)
    # replay context and replay: arguments and shapes before any CUDA call
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_abft_capture(0, 4096, 8192, 128, 256, 64, 12288, 0, 4, 16384, 20480, 24576, 0, 0, 0, 0, 28672, 0)
    assert ei.value.status == 1
    for M, N, K in [(0, 256, 64), (128, 260, 64), (128, 256, 60)]:
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_capture(4096, 8192, 12288, M, N, K, 16384, 0, 4, 16384, 20480, 24576, 0, 0, 0, 0, 28672, 0)
        assert ei.value.status == 9, (M, N, K)
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_capture_wgrad(4096, 8192, 12288, M, N, K, 16384, 0, 4, 16384, 20480, 24576, 0, 0, 0, 0,
                                       28672, 0)
        assert ei.value.status == 9, (M, N, K)
    with pytest.raises(sdc.SdcError) as ei:  # a cap with no buffer
        sdc.sdc_abft_capture(4096, 8192, 12288, 128, 256, 64, 16384, 0, 4, 0, 0, 0, 0, 0, 0, 0, 28672, 0)
    assert ei.value.status == 1
    for cap, N, K in [(0, 256, 64), (1025, 256, 64), (4, 260, 64)]:
        assert sdc.sdc_abft_replay_workspace_size(cap, N, K) == 0
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_replay(4096, N, K, cap, 8192, 12288, 16384, 20480, 24576, 28672, 32768, 1 << 20, 0)
        assert ei.value.status == 9, (cap, N, K)
    for T, cr, cc in [(0, 4, 4), (128, 0, 4), (128, 4, 65)]:
        assert sdc.sdc_abft_replay_wgrad_workspace_size(T, cr, cc) == 0
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_replay_wgrad(T, 256, 64, cr, cc, *[4096 * (i + 1) for i in range(10)], 1 << 20, 0)
        assert ei.value.status == 9, (T, cr, cc)
    for K, cr, cc in [(0, 4, 4), (60, 4, 4), (64, 0, 4), (64, 4, 65)]:
        assert sdc.sdc_abft_replay_pairs_workspace_size(K, cr, cc) == 0
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_abft_replay_pairs(128, 256, K, cr, cc, *[4096 * (i + 1) for i in range(10)], 1 << 20, 0)
        assert ei.value.status == 9, (K, cr, cc)
    # staged A rows (cap_r x 128 of K) and W rows (cap_c x 256 of K), the replayed C, its row checksums, the
    # abort word, a GEMM's workspace
    assert sdc.sdc_abft_replay_pairs_workspace_size(64, 1, 1) == (128 * 64 * 2 + 256 * 64 * 2 + 128 * 256 * 2
                                                                  + 1024 + 256 + sdc.sdc_abft_workspace_size(128, 256, 64))
    # staged rows (cap x 128 rows of K and of N bf16), their row checksums, the abort word, a GEMM's workspace
    assert sdc.sdc_abft_replay_workspace_size(1, 256, 64) == (128 * 64 * 2 + 128 * 256 * 2 + 1024 + 256
                                                              + sdc.sdc_abft_workspace_size(128, 256, 64))
    assert sdc.sdc_abft_replay_wgrad_workspace_size(512, 2, 1) == (
        512 * 256 * 2 + 512 * 256 * 2 + 256 * 256 * 2 + 256 * 8 + 256 + sdc.sdc_abft_wgrad_workspace_size(512, 256, 256))
    # bounded-wait self-test: arguments checked before the launch
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_selftest_bounded_wait(10, 0, 0)
    assert ei.value.status == 1
    for polls in (0, 1 << 25):
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_selftest_bounded_wait(polls, 4096, 0)
        assert ei.value.status == 9
    # attention invariant: inputs checked, then shapes and scalars, before any CUDA call
    fake = [4096, 8192, 12288, 16384]
    outs = [20480 + 4096 * i for i in range(8)]
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_attn_dv_check(0, *fake[1:], 1, 128, 128, 0.088, 0, 1.0, *outs, 0, 0, 0)
    assert ei.value.status == 1
    for BH, L, D, scale, causal, tol in [(1, 128, 64, 0.088, 0, 1.0), (1, 102, 128, 0.088, 0, 1.0), (1, 0, 128, 0.088, 0, 1.0),
                                         (0, 128, 128, 0.088, 0, 1.0), (1, 128, 128, -1.0, 0, 1.0),
                                         (1, 128, 128, 0.088, 2, 1.0), (1, 128, 128, 0.088, 0, 0.0)]:
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_attn_dv_check(*fake, BH, L, D, scale, causal, tol, *outs, 0, 0, 0)
        assert ei.value.status == 9, (BH, L, D, scale, causal, tol)
    # dO partials (float4 per block and column), dV partials (float2), lse log2(e) (a float
    # per token), the abort word and the counters (16 bytes + one word per head, in 256-byte units)
    assert sdc.sdc_attn_workspace_size(2, 256, 128) == (2 * 2 * 128 * 16 + 2 * 2 * 128 * 8 + 2 * 256 * 4 + 256)
    assert sdc.sdc_attn_workspace_size(64, 128, 128) == (64 * 128 * 16 + 64 * 128 * 8 + 64 * 128 * 4 + 512)
    # a partial last block counts as a block: 100 tokens take one block of partials
    assert sdc.sdc_attn_workspace_size(2, 100, 128) == (2 * 128 * 16 + 2 * 128 * 8 + 256 * ((2 * 100 * 4 + 255) // 256) + 256)
    assert sdc.sdc_attn_workspace_size(2, 256, 64) == 0
    # grouped attention: group 0, or a group that does not divide the query heads, is rejected
    outs = [4096] * 8
    for BH, group in [(4, 0), (6, 4), (2, 3)]:
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_attn_dv_check_grouped(4096, 8192, 16384, 32768, BH, group, 128, 128, 0.088, 0, 1.0, *outs,
                                          0, 0, 0)
        assert ei.value.status == 9, (BH, group)
    # one work item's steps, group x ceil(L / 128), at most 2^19 (the epilogue's bounded wait)
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_attn_dv_check_grouped(4096, 8192, 16384, 32768, 1024, 1024, 65536 + 128, 128, 0.088, 0, 1.0, *outs,
                                      0, 0, 0)
    assert ei.value.status == 9
    assert sdc.sdc_abft_workspace_size(128, 16384, 64) == (64 * 128 * 8 + 1 * 16384 * 8 + 2 * 512 + (64 + 16) * 64 * 16
                                                           + (128 + 16384) * 16 + 2304 + 256)


def test_pages_verdict_decoding(sdc):
    assert sdc.pages_verdict({"diverged": 0, "no_majority": 0, "suspect_mask": 0}) == \
        {"diverged": False, "suspects": []}
    assert sdc.pages_verdict({"diverged": 1, "no_majority": 1, "suspect_mask": 4}) == \
        {"diverged": True, "suspects": None}
    assert sdc.pages_verdict({"diverged": 1, "no_majority": 0, "suspect_mask": 0b1010}) == \
        {"diverged": True, "suspects": [1, 3]}
    raw = np.zeros(1, dtype=sdc.VOTE_SUMMARY_DTYPE)
    raw["diverged"] = 1
    raw["suspect_mask"] = 1 << 63
    assert sdc.decode_summary(raw.view(np.uint8))["suspect_mask"] == 1 << 63


def test_binding_signatures_match_header(sdc):
    # every entry point of include/sdc.h has a ctypes signature of the same arity
    import silent_corruption_checksums_gb300 as m
    hdr = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = re.findall(r"\n(?:sdc_status|size_t|const char \*|void)\s+\*?(sdc_\w+)\s*\(([^;]*?)\);", hdr)
    assert len(decls) >= 20
    lib = m._load()
    for name, args in decls:
        n_c = 0 if args.strip() in ("", "void") else args.count(",") + 1
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == n_c, (name, n_c, len(fn.argtypes))


def test_header_compiles_alone_and_layouts_match_binding(sdc, tmp_path):
    """include/sdc.h compiled as C11 on its own (no CUDA header on the path, warnings as errors): every
    struct's size and field offsets, the dtype codes and the limits equal the Python binding's."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")

    def np_layout(dt):
        return dt.itemsize, {n: dt.fields[n][1] for n in dt.names}

    def ct_layout(cls):
        return ctypes.sizeof(cls), {n: getattr(cls, n).offset for n, _ in cls._fields_}

    expect = {
        "sdc_tensor_desc": np_layout(sdc.DESC_DTYPE),
        "sdc_grad_stats": np_layout(sdc.GRAD_STATS_DTYPE),
        "sdc_vote_summary": np_layout(sdc.VOTE_SUMMARY_DTYPE),
        "sdc_ring_summary": np_layout(sdc.RING_SUMMARY_DTYPE),
        "sdc_adamw_hparams": ct_layout(sdc.AdamWHparams),
        "sdc_plan_opts": ct_layout(sdc._PlanOpts),
        "sdc_abft_summary": (8, {"n_flagged": 0, "n_flagged_cols": 4}),  # read as int32[2] by the binding
    }
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "sdc.h"', "int main(void) {"]
    for s, (_, fields) in expect.items():
        lines.append(f'    printf("S {s} %zu\\n", sizeof({s}));')
        for f in fields:
            lines.append(f'    printf("F {s} {f} %zu\\n", offsetof({s}, {f}));')
    statuses = ["SDC_OK", "SDC_ERR_NULL", "SDC_ERR_BAD_ELEM_SIZE", "SDC_ERR_SHAPE_MISMATCH", "SDC_ERR_TOO_MANY_REPLICAS",
                "SDC_ERR_WS_TOO_SMALL", "SDC_ERR_CUDA", "SDC_ERR_BAD_DTYPE", "SDC_ERR_BAD_POINTER", "SDC_ERR_BAD_ARG",
                "SDC_ERR_WRONG_DEVICE"]
    for c in statuses + ["SDC_DTYPE_RAW", "SDC_DTYPE_F32", "SDC_DTYPE_BF16", "SDC_DTYPE_F16", "SDC_MAX_REPLICAS"]:
        lines.append(f'    printf("C {c} %lu\\n", (unsigned long)({c}));')
    lines.append('    printf("C SDC_NOALLOC_SCRATCH_BYTES %lu\\n", (unsigned long)(SDC_NOALLOC_SCRATCH_BYTES));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe)], check=True)
    got_size, got_off, consts = {}, {}, {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        f = line.split()
        if f[0] == "S":
            got_size[f[1]] = int(f[2])
        elif f[0] == "F":
            got_off[(f[1], f[2])] = int(f[3])
        else:
            consts[f[1]] = int(f[2])
    for s, (size, fields) in expect.items():
        assert got_size[s] == size, s
        for f, off in fields.items():
            assert got_off[(s, f)] == off, (s, f)
    assert [consts[k] for k in ("SDC_DTYPE_RAW", "SDC_DTYPE_F32", "SDC_DTYPE_BF16", "SDC_DTYPE_F16")] == \
        [sdc.DTYPE_RAW, sdc.DTYPE_F32, sdc.DTYPE_BF16, sdc.DTYPE_F16]
    assert consts["SDC_MAX_REPLICAS"] == sdc.MAX_REPLICAS
    for name in statuses:  # each status code's string is its name in the header
        assert sdc.sdc_status_string(consts[name]) == name
    assert consts["SDC_NOALLOC_SCRATCH_BYTES"] == sdc.NOALLOC_SCRATCH_BYTES
