"""The tensor-core checks inside a CUDA graph and on concurrent streams.

The GEMM with row + column checksums and the attention invariant reset their own
counters with memset nodes and launch persistent kernels (one over a banded tile
schedule, one with a work queue): captured once and replayed, and run at the same time
on two streams with their own workspaces, they give results bit-identical to eager
calls on the same inputs, and a replay after an in-place change of an input reads
the new values.  The same holds for the weight-gradient GEMM with its check and for a
plan's xorsum with the pair compare (the launches the benchmark replays from graphs).
"""
import pytest
import torch

import sdc_workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
GEMM = (512, 1024, 1024)
ATTN = (4, 1024)


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _outs_gemm(g):
    return [g.C, g.rowsum, g.colsum, g.residual, g.bound, g.flag, g.residual_col, g.bound_col, g.flag_col,
            g.summary, g.aborted]


def _outs_attn(a):
    return [a.dV, a.colsum_dv, a.colsum_do, a.residual, a.bound, a.flag, a.summary, a.aborted]


def _bits(ts):
    return [t.contiguous().view(torch.uint8).clone() for t in ts]


def _same(xs, ys):
    for i, (x, y) in enumerate(zip(xs, ys)):
        assert torch.equal(x, y), i


def _inputs():
    ops = W.gemm_operands(*GEMM, DEV, seed=51)
    x = W.attn_inputs(*ATTN, DEV, seed=52, causal=True)
    return ops, x


def _eager(sdc, ops, x):
    g = sdc.AbftGemm(*GEMM, DEV, columns=True)
    a = sdc.AttnDvCheck(*ATTN, DEV)
    g(ops["A"], ops["W"])
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True)
    torch.cuda.synchronize()
    assert int(g.aborted[0]) == 0 and int(a.aborted[0]) == 0
    assert int(g.summary[0]) == 0 and int(g.summary[1]) == 0 and int(a.summary[0]) == 0
    return _bits(_outs_gemm(g)), _bits(_outs_attn(a))


def test_checks_in_a_cuda_graph(sdc):
    ops, x = _inputs()
    ref_g, ref_a = _eager(sdc, ops, x)
    g = sdc.AbftGemm(*GEMM, DEV, columns=True)
    a = sdc.AttnDvCheck(*ATTN, DEV)
    s = torch.cuda.Stream()

    def work():
        g(ops["A"], ops["W"], stream=s)
        a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True, stream=s)

    with torch.cuda.stream(s):
        work()  # warm up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        work()
    for t in _outs_gemm(g) + _outs_attn(a):
        t.zero_()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        _same(_bits(_outs_gemm(g)), ref_g)
        _same(_bits(_outs_attn(a)), ref_a)
    # change inputs in place: the next replay reads them (compared with eager calls on the same data)
    W.xor_element(ops["A"], 7 * GEMM[2] + 3, 0x4000)
    W.xor_element(x["K"], 2 * ATTN[1] * 128 + 5 * 128 + 17, 0x4000)
    graph.replay()
    torch.cuda.synchronize()
    got_g, got_a = _bits(_outs_gemm(g)), _bits(_outs_attn(a))
    e = sdc.AbftGemm(*GEMM, DEV, columns=True)
    f = sdc.AttnDvCheck(*ATTN, DEV)
    e(ops["A"], ops["W"])
    f(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True)
    torch.cuda.synchronize()
    _same(got_g, _bits(_outs_gemm(e)))
    _same(got_a, _bits(_outs_attn(f)))
    assert not torch.equal(got_g[0], ref_g[0]) and not torch.equal(got_a[0], ref_a[0])
    assert int(f.summary[0]) > 0  # the corrupted key breaks the invariant of some columns


def test_two_streams_at_once(sdc):
    ops, x = _inputs()
    ref_g, ref_a = _eager(sdc, ops, x)
    g = sdc.AbftGemm(*GEMM, DEV, columns=True)
    a = sdc.AttnDvCheck(*ATTN, DEV)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        g(ops["A"], ops["W"], stream=s1)
        a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True, stream=s2)
    torch.cuda.synchronize()
    _same(_bits(_outs_gemm(g)), ref_g)
    _same(_bits(_outs_attn(a)), ref_a)


def test_wgrad_check_and_xorsum_pairs_in_a_cuda_graph(sdc):
    # the weight-gradient GEMM and its check, and a plan's xorsum with the pair compare, captured once:
    # replays are bit-identical to eager calls, and read inputs changed in place
    T, N, K = 1024, 512, 768
    ops = W.wgrad_operands(T, N, K, DEV, seed=55)
    rng_tensors = [W.gemm_operands(8, 8 * (i + 1), 64, DEV, seed=56 + i)["W"] for i in range(5)]  # [8 (i + 1), 64]
    copies = [t.clone() for t in rng_tensors]
    W.xor_element(copies[3], 17, 0x0100)
    e = sdc.AbftWgrad(T, N, K, DEV)
    e(ops["dY"], ops["X"])
    ep = sdc.Plan([rng_tensors, copies])
    ex = ep.xorsum()
    em, ed = sdc.xorsum_compare(ex[0], ex[1])
    torch.cuda.synchronize()
    outs = lambda a: [a.dW, a.rowsum, a.colsum, a.residual, a.bound, a.flag, a.residual_col, a.bound_col,
                      a.flag_col, a.summary, a.aborted]
    ref = _bits(outs(e)) + _bits([ex, em, ed])
    a = sdc.AbftWgrad(T, N, K, DEV)
    plan = sdc.Plan([rng_tensors, copies])
    xo = torch.empty((2, 5), dtype=torch.int64, device=DEV)
    s = torch.cuda.Stream()
    res = {}

    def work():
        a(ops["dY"], ops["X"], stream=s)
        plan.xorsum(out=xo, stream=s)
        res["m"], res["d"] = sdc.xorsum_compare(xo[0], xo[1], stream=s)

    with torch.cuda.stream(s):
        work()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        work()
    for t in outs(a) + [xo]:
        t.zero_()
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        _same(_bits(outs(a)) + _bits([xo, res["m"], res["d"]]), ref)
    assert int(res["m"].sum()) == 1 and int(res["m"][3]) == 1
    W.xor_element(copies[1], 5, 0x0001)  # a second pair now differs
    graph.replay()
    torch.cuda.synchronize()
    assert res["m"].cpu().tolist() == [0, 1, 0, 1, 0]
