"""Every output array and workspace a call is given is checked on the host
before anything is enqueued: memory that is not device memory of the current
device, or a range that runs past its allocation, is SDC_ERR_BAD_POINTER (8).

Each case first makes the call with valid arguments, then with one output
replaced by host memory (a CPU tensor) or sized past a small allocation; the
rejected call must leave the device untouched.
"""
import pytest
import torch

import sdc_workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BAD_POINTER = 8
_held = []  # host tensors whose addresses the calls are given, kept alive until the module ends


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    yield m
    _held.clear()


def _host(n_bytes, align=1):
    """Address of n_bytes of host (pageable) memory, aligned to `align`."""
    t = torch.zeros(n_bytes + align + 8, dtype=torch.uint8)
    _held.append(t)
    return (t.data_ptr() + align - 1) // align * align


def _rejects(fn, *args):
    import silent_corruption_checksums_gb300 as m
    with pytest.raises(m.SdcError) as ei:
        fn(*args)
    assert ei.value.status == BAD_POINTER, str(ei.value)


def test_fingerprint_xorsum_vote_outputs(sdc):
    ts = [torch.arange(1000, dtype=torch.int32, device=DEV), torch.ones(77, dtype=torch.uint8, device=DEV)]
    plan = sdc.Plan([ts, [t.clone() for t in ts], [t.clone() for t in ts]])
    R, T = 3, 2
    out = torch.empty((R, T, 2), dtype=torch.int64, device=DEV)
    ws, wsb = plan.ws.data_ptr(), plan.ws_bytes
    sdc.sdc_fingerprint(plan.handle, out.data_ptr(), ws, wsb, 0)
    _rejects(sdc.sdc_fingerprint, plan.handle, _host(R * T * 16), ws, wsb, 0)
    _rejects(sdc.sdc_fingerprint, plan.handle, out.data_ptr(), _host(wsb, 256), wsb, 0)
    xo = torch.empty((R, T), dtype=torch.int64, device=DEV)
    sdc.sdc_xorsum(plan.handle, xo.data_ptr(), ws, wsb, 0)
    _rejects(sdc.sdc_xorsum, plan.handle, _host(R * T * 8), ws, wsb, 0)

    mism = torch.empty(T, dtype=torch.uint8, device=DEV)
    diff = torch.empty(T, dtype=torch.int64, device=DEV)
    sdc.sdc_xorsum_compare(xo[0].data_ptr(), xo[1].data_ptr(), T, mism.data_ptr(), diff.data_ptr(), 0)
    _rejects(sdc.sdc_xorsum_compare, xo[0].data_ptr(), xo[1].data_ptr(), T, _host(T), diff.data_ptr(), 0)
    _rejects(sdc.sdc_xorsum_compare, xo[0].data_ptr(), xo[1].data_ptr(), T, mism.data_ptr(), _host(8 * T), 0)

    suspect = torch.empty(T, dtype=torch.int32, device=DEV)
    mask = torch.empty(T, dtype=torch.int64, device=DEV)
    summ = torch.zeros(24, dtype=torch.uint8, device=DEV)
    sdc.sdc_vote(out.data_ptr(), R, T, suspect.data_ptr(), mask.data_ptr(), summ.data_ptr(), 0)
    _rejects(sdc.sdc_vote, out.data_ptr(), R, T, suspect.data_ptr(), mask.data_ptr(), _host(24), 0)
    _rejects(sdc.sdc_vote, out.data_ptr(), R, T, _host(4 * T), mask.data_ptr(), summ.data_ptr(), 0)
    # a table of 10^8 tensors read from a 96-byte allocation runs past it
    _rejects(sdc.sdc_vote, out.data_ptr(), R, 10 ** 8, suspect.data_ptr(), mask.data_ptr(), summ.data_ptr(), 0)
    torch.cuda.synchronize()
    assert int(summ[0]) == 0  # the valid vote: all replicas agree


def test_grad_outputs(sdc):
    g = [torch.randn(4096, device=DEV).to(torch.bfloat16) for _ in range(2)]
    avg = torch.empty_like(g[0])
    pre = torch.empty((2, 56), dtype=torch.uint8, device=DEV)
    post = torch.empty(56, dtype=torch.uint8, device=DEV)
    n = g[0].numel()
    wsb = sdc.sdc_grad_average_scan_workspace_size(n, 2, 2)
    ws = torch.empty(wsb + 256, dtype=torch.uint8, device=DEV)
    wsp = (ws.data_ptr() + 255) // 256 * 256
    bufs = [t.data_ptr() for t in g]
    sdc.sdc_grad_average_scan(bufs, avg.data_ptr(), n, 2, pre.data_ptr(), post.data_ptr(), wsp, wsb, 0)
    _rejects(sdc.sdc_grad_average_scan, bufs, avg.data_ptr(), n, 2, _host(112), post.data_ptr(), wsp, wsb, 0)
    _rejects(sdc.sdc_grad_average_scan, bufs, avg.data_ptr(), n, 2, pre.data_ptr(), _host(56), wsp, wsb, 0)
    _rejects(sdc.sdc_grad_average_scan, bufs, avg.data_ptr(), n, 2, pre.data_ptr(), post.data_ptr(), _host(wsb, 256),
             wsb, 0)
    # the no-allocation entry point still accepts its own static scratch
    sdc.sdc_grad_average_scan_noalloc(bufs, avg.data_ptr(), n, 2, pre.data_ptr(), post.data_ptr(), 0)

    plan = sdc.Plan([[g[0]], [g[1]]])
    stats = torch.empty((2, 56), dtype=torch.uint8, device=DEV)
    sdc.sdc_grad_scan(plan.handle, stats.data_ptr(), plan.ws.data_ptr(), plan.ws_bytes, 0)
    _rejects(sdc.sdc_grad_scan, plan.handle, _host(112), plan.ws.data_ptr(), plan.ws_bytes, 0)
    torch.cuda.synchronize()
    assert sdc.decode_stats(stats)[0]["n_nan"] == 0


def test_ring_and_selftest_outputs(sdc):
    n, L = 4, 3
    table = torch.zeros((n, 2, L), dtype=torch.int64, device=DEV)
    mism = torch.empty(n, dtype=torch.uint8, device=DEV)
    hits = torch.empty(n, dtype=torch.int32, device=DEV)
    culprit = torch.empty(n, dtype=torch.uint8, device=DEV)
    amb = torch.empty(n, dtype=torch.uint8, device=DEV)
    summ = torch.empty(4, dtype=torch.int32, device=DEV)
    args = [table.data_ptr(), n, L, 1, mism.data_ptr(), hits.data_ptr(), culprit.data_ptr(), amb.data_ptr(),
            summ.data_ptr(), 0]
    sdc.sdc_ring_audit(*args)
    for pos, size in ((5, 4 * n), (8, 16)):
        bad = list(args)
        bad[pos] = _host(size)
        _rejects(sdc.sdc_ring_audit, *bad)
    _rejects(sdc.sdc_selftest_bounded_wait, 16, _host(4), 0)
    torch.cuda.synchronize()
    assert int(summ[1]) == 0


def test_abft_outputs(sdc):
    M, N, K = 128, 256, 64
    ops = W.gemm_operands(M, N, K, DEV, seed=31)
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    A, Wt = ops["A"].data_ptr(), ops["W"].data_ptr()
    gemm = [A, Wt, g.C.data_ptr(), M, N, K, g.rowsum.data_ptr(), g.colsum.data_ptr(), g.aborted.data_ptr(),
            g.ws.data_ptr(), g.ws_bytes, 0]
    sdc.sdc_abft_gemm(*gemm)
    for pos, size in ((6, 8 * M), (7, 8 * N), (8, 4)):
        bad = list(gemm)
        bad[pos] = _host(size)
        _rejects(sdc.sdc_abft_gemm, *bad)
    verify = [A, Wt, M, N, K, g.rowsum.data_ptr(), g.colsum.data_ptr(), 1.0, g.residual.data_ptr(),
              g.bound.data_ptr(), g.flag.data_ptr(), g.residual_col.data_ptr(), g.bound_col.data_ptr(),
              g.flag_col.data_ptr(), g.summary.data_ptr(), g.ws.data_ptr(), g.ws_bytes, 0]
    sdc.sdc_abft_verify(*verify)
    for pos, size in ((8, 8 * M), (9, 8 * M), (10, M), (11, 8 * N), (12, 8 * N), (13, N), (14, 8)):
        bad = list(verify)
        bad[pos] = _host(size)
        _rejects(sdc.sdc_abft_verify, *bad)
    torch.cuda.synchronize()
    assert int(g.aborted[0]) == 0 and int(g.summary[0]) == 0 and int(g.summary[1]) == 0


def test_attention_outputs(sdc):
    BH, L = 2, 256
    x = W.attn_inputs(BH, L, DEV, seed=33, causal=True)
    chk = sdc.AttnDvCheck(BH, L, DEV)
    args = [x["Q"].data_ptr(), x["K"].data_ptr(), x["dO"].data_ptr(), x["lse"].data_ptr(), BH, 1, L, 128,
            x["scale"], 1, 1.0, chk.dV.data_ptr(), chk.colsum_dv.data_ptr(), chk.colsum_do.data_ptr(),
            chk.residual.data_ptr(), chk.bound.data_ptr(), chk.flag.data_ptr(), chk.summary.data_ptr(),
            chk.aborted.data_ptr(), chk.ws.data_ptr(), chk.ws_bytes, 0]
    sdc.sdc_attn_dv_check_grouped(*args)
    col = BH * 128
    for pos, size in ((12, 8 * col), (13, 8 * col), (14, 8 * col), (15, 8 * col), (16, col), (17, 8), (18, 4)):
        bad = list(args)
        bad[pos] = _host(size)
        _rejects(sdc.sdc_attn_dv_check_grouped, *bad)
    bad = list(args)
    bad[19] = _host(chk.ws_bytes, 256)
    _rejects(sdc.sdc_attn_dv_check_grouped, *bad)
    torch.cuda.synchronize()
    assert int(chk.aborted[0]) == 0 and int(chk.summary[0]) == 0
