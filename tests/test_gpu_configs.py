"""The five workloads at full size, in the launch configuration the benchmark
times, checked against the oracle (whole workloads where the host can redo
them in seconds, sampled tensors plus ground truth elsewhere)."""
import os

import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import assert_attn_bound, assert_verifier_bound, assert_wgrad_bound, fp_table, host_bits, stats_match

pytestmark = [pytest.mark.gpu, pytest.mark.big]
DEV = "cuda"
THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _vote(sdc, fp):
    suspect, mask, summary = sdc.vote(fp)
    return suspect.cpu().tolist(), mask.cpu().numpy().view(np.uint64).tolist(), sdc.decode_summary(summary)


def test_tiny_config(sdc):
    w = W.tiny(DEV, seed=0)
    plan = sdc.Plan(w["replicas"])
    fp = plan.fingerprint()
    got = fp_table(fp)
    ref = [[oracle.fingerprint(host_bits(t)) for t in ts] for ts in w["replicas"]]
    assert got == ref
    s, m, summ = _vote(sdc, fp)
    rs, rm, rsumm = oracle.vote(ref)
    assert s == rs and m == rm and sdc.pages_verdict(summ) == oracle.pages_verdict(rsumm) == \
        {"diverged": True, "suspects": [1]}


def test_1b_fp32_three_replicas_full_oracle(sdc):
    w = W.weights_1b(DEV, seed=1)
    plan = sdc.Plan(w["replicas"])
    fp = plan.fingerprint()
    got = fp_table(fp)
    ref = [[oracle.fingerprint(host_bits(t), threads=THREADS) for t in ts] for ts in w["replicas"]]
    assert got == ref
    t = w["truth"]
    s, m, summ = _vote(sdc, fp)
    rs, rm, rsumm = oracle.vote(ref)
    assert s == rs and m == rm
    exp = [-1] * len(w["layout"])
    exp[t["tensor"]] = t["replica"]
    assert s == exp
    assert sdc.pages_verdict(summ) == {"diverged": True, "suspects": [t["replica"]]}
    xs = plan.xorsum().cpu().numpy().view(np.uint64)
    for r in range(3):
        assert int(xs[r, t["tensor"]]) == oracle.xorsum(host_bits(w["replicas"][r][t["tensor"]]), threads=THREADS)


def test_grad_config_full_oracle(sdc):
    g = W.grads_1b(DEV, seed=3)
    bufs = g["bufs"]
    avg, pre, post = sdc.grad_average_scan(bufs)
    torch.cuda.synchronize()
    hb = [host_bits(b) for b in bufs]
    got_pre = sdc.decode_stats(pre)
    for b in range(4):
        stats_match(got_pre[b], oracle.grad_stats(hb[b], "bf16", threads=THREADS))
    # ground truth of the injector: counts of the injected buffer
    kinds = [k for _, k in g["truth"]]
    assert got_pre[2]["n_nan"] == kinds.count("nan")
    assert got_pre[2]["n_inf"] == kinds.count("+inf") + kinds.count("-inf")
    assert got_pre[2]["n_big"] == kinds.count("+2^70") + kinds.count("-2^70")
    ref_avg = oracle.average(hb, "bf16", threads=THREADS)
    assert np.array_equal(host_bits(avg), ref_avg)
    got_post = sdc.decode_stats(post)[0]
    stats_match(got_post, oracle.grad_stats(ref_avg, "bf16", threads=THREADS))
    assert got_post["nonfinite_fp32"] == 1


def test_8b_bf16_eight_replicas_sampled(sdc):
    w = W.weights_8b(DEV, seed=4)
    reps = w["replicas"]
    plan = sdc.Plan(reps)
    fp = plan.fingerprint()
    got = fp_table(fp)
    t = w["truth"]
    k = t["tensor"]
    for r in range(8):  # every copy of the perturbed tensor
        assert got[r][k] == oracle.fingerprint(host_bits(reps[r][k]), threads=THREADS)
    rng = np.random.default_rng(40)
    for _ in range(8):  # random other copies
        r, kk = int(rng.integers(8)), int(rng.integers(len(reps[0])))
        assert got[r][kk] == oracle.fingerprint(host_bits(reps[r][kk]), threads=THREADS)
    s, m, summ = _vote(sdc, fp)
    exp = [-1] * len(w["layout"])
    exp[k] = t["replica"]
    assert s == exp and m[k] == 1 << t["replica"]
    assert sdc.pages_verdict(summ) == {"diverged": True, "suspects": [t["replica"]]}
    # property at any size: the copies that were not touched agree exactly
    for kk in range(len(reps[0])):
        if kk != k:
            assert len({got[r][kk] for r in range(8)}) == 1


def test_stress_many_small_tensors_sampled(sdc):
    w = W.stress(DEV, seed=5)
    reps = w["replicas"]
    plan = sdc.Plan(reps)
    fp = plan.fingerprint()
    got = fp_table(fp)
    t = w["truth"]
    T = len(reps[0])
    for r in range(3):
        assert got[r][t["tensor"]] == oracle.fingerprint(host_bits(reps[r][t["tensor"]]))
    rng = np.random.default_rng(50)
    for _ in range(1500):
        r, k = int(rng.integers(3)), int(rng.integers(T))
        assert got[r][k] == oracle.fingerprint(host_bits(reps[r][k])), (r, k)
    s, m, summ = _vote(sdc, fp)
    assert [i for i, v in enumerate(s) if v != -1] == [t["tensor"]]
    assert s[t["tensor"]] == t["replica"]
    assert sdc.pages_verdict(summ) == {"diverged": True, "suspects": [t["replica"]]}
    # grad statistics over a seeded sample of 5,000 mixed-dtype tensors (counts exact, norm to 1e-10)
    names = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}
    idx = np.sort(rng.choice(T, size=5000, replace=False))
    sub = [reps[0][i] for i in idx]
    gplan = sdc.Plan([sub])
    stats = sdc.decode_stats(gplan.grad_scan())
    ref0 = oracle.grad_stats_multi([host_bits(x) for x in sub], [names[x.dtype] for x in sub], threads=THREADS)
    stats_match(stats[0], ref0)
    # xorsum compare of 1,000 (original, recomputed) pairs
    p = w["pairs"]
    pplan = sdc.Plan([p["orig"], p["recomp"]])
    xs = pplan.xorsum()
    mism, diff = sdc.xorsum_compare(xs[0], xs[1])
    xs_np = xs.cpu().numpy().view(np.uint64)
    for i in range(len(p["orig"])):
        assert int(xs_np[0, i]) == oracle.xorsum(host_bits(p["orig"][i]))
        assert int(xs_np[1, i]) == oracle.xorsum(host_bits(p["recomp"][i]))
    differ = {i for i, _, _ in p["differ"]}
    assert set(np.nonzero(mism.cpu().numpy())[0].tolist()) == differ
    dnp = diff.cpu().numpy().view(np.uint64)
    for i, e, b in p["differ"]:
        assert int(dnp[i]) == 1 << b


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_gemm_checksum_bench_shape(sdc):
    # the benchmark's GEMM (8b MLP up-projection, 8192 x 14336 x 4096, rows + columns, the same
    # seed) in its launch configuration; sampled rows and columns against the oracle one by one
    M, N, K = W.GEMM_8B_UP
    ops = W.gemm_operands(M, N, K, DEV, seed=6)
    g = sdc.AbftGemm(M, N, K, DEV, columns=True)
    g(ops["A"], ops["W"])
    torch.cuda.synchronize()
    assert int(g.aborted[0]) == 0
    assert int(g.summary[0]) == 0 and int(g.summary[1]) == 0  # no clean row or column flagged
    A64 = oracle.bf16_to_f64(_bf16_bits(ops["A"]))
    W64 = oracle.bf16_to_f64(_bf16_bits(ops["W"]))
    rng = np.random.default_rng(61)
    gk = K * 2.0 ** -22
    rows = np.sort(rng.choice(M, 12, replace=False))
    exact = A64[rows] @ W64.T
    e = gk * (1 + gk) * (np.abs(A64[rows]) @ np.abs(W64).T) + 2.0 * K * 2.0 ** -126
    C = g.C[torch.as_tensor(rows, device=DEV)].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(C - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134)
    mag_r = np.abs(A64[rows]) @ np.abs(W64).sum(axis=0)
    bound_r = oracle.abft_bound(mag_r, N, K)
    rs = g.rowsum.cpu().numpy()[rows]
    assert np.all(np.abs(rs - exact.sum(axis=1)) <= bound_r)
    assert_verifier_bound(g.bound.cpu().numpy()[rows], bound_r, mag_r, N, K)
    cols = np.sort(rng.choice(N, 8, replace=False))
    exact_c = (A64 @ W64[cols].T).sum(axis=0)
    bound_c = oracle.abft_bound(np.abs(W64[cols]) @ np.abs(A64).sum(axis=0), M, K)
    assert np.all(np.abs(g.colsum.cpu().numpy()[cols] - exact_c) <= bound_c)


def test_wgrad_checksum_bench_shape(sdc):
    # the benchmark's weight gradient (dW = dY^T X, 8192 tokens, dY [8192, 14336], X [8192, 4096],
    # rows + columns, the same seed) in its launch configuration; sampled rows and columns of dW
    # against the oracle one by one, no flag anywhere
    T, N, K = W.GEMM_8B_UP
    ops = W.wgrad_operands(T, N, K, DEV, seed=10)
    a = sdc.AbftWgrad(T, N, K, DEV)
    a(ops["dY"], ops["X"])
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0 and int(a.summary[1]) == 0
    dY64 = oracle.bf16_to_f64(_bf16_bits(ops["dY"]))
    X64 = oracle.bf16_to_f64(_bf16_bits(ops["X"]))
    ra, qa = np.abs(X64).sum(axis=1), np.abs(dY64).sum(axis=1)  # per token: sum |X|, sum |dY|
    rng = np.random.default_rng(62)
    g = T * 2.0 ** -22
    rows = np.sort(rng.choice(N, 12, replace=False))
    exact = dY64[:, rows].T @ X64  # rows of dW [12, K]
    e = g * (1 + g) * (np.abs(dY64[:, rows]).T @ np.abs(X64)) + 2.0 * T * 2.0 ** -126
    dW = a.dW[torch.as_tensor(rows, device=DEV)].float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(dW - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134)
    mag_r = np.abs(dY64[:, rows]).T @ ra
    bound_r = oracle.abft_bound(mag_r, K, T)
    assert np.all(np.abs(a.rowsum.cpu().numpy()[rows] - exact.sum(axis=1)) <= bound_r)
    assert_wgrad_bound(a.bound.cpu().numpy()[rows], bound_r, mag_r, K, T)
    cols = np.sort(rng.choice(K, 8, replace=False))
    exact_c = (dY64.T @ X64[:, cols]).sum(axis=0)
    mag_c = np.abs(X64[:, cols]).T @ qa
    bound_c = oracle.abft_bound(mag_c, N, T)
    assert np.all(np.abs(a.colsum.cpu().numpy()[cols] - exact_c) <= bound_c)
    assert_wgrad_bound(a.bound_col.cpu().numpy()[cols], bound_c, mag_c, N, T)


def test_attention_invariant_bench_shape(sdc):
    # the benchmark's attention backward (32 heads x 4096 x 128, causal, the same seed) in its
    # launch configuration; two sampled heads in full against the oracle, no flag anywhere
    BH, L = W.ATTN_8B
    x = W.attn_inputs(BH, L, DEV, seed=8, causal=True)
    a = sdc.AttnDvCheck(BH, L, DEV)
    a(x["Q"], x["K"], x["dO"], x["lse"], x["scale"], True)
    torch.cuda.synchronize()
    assert int(a.aborted[0]) == 0 and int(a.summary[0]) == 0
    g = L * 2.0 ** -22
    eps = 2.0 ** -8 * (1 + 2.0 ** -7) + g * (1 + g) * (1 + 2.0 ** -7)
    for h in (0, 19):
        Qb, Kb, dOb = (_bf16_bits(x[k][h]) for k in ("Q", "K", "dO"))
        P = oracle.attn_probs(Qb, Kb, x["lse"][h].cpu().numpy(), x["scale"], True)
        exact = oracle.attn_dv(P, dOb)
        e = eps * (P.T @ np.abs(oracle.bf16_to_f64(dOb)))
        dV = a.dV[h].float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(dV - exact) <= 2.0 ** -8 * (np.abs(exact) + e) + e + 2.0 ** -134)
        v = oracle.attn_invariant(a.colsum_dv[h].cpu().numpy(), dOb)
        assert v["n_flagged"] == 0
        assert np.all(np.abs(a.colsum_dv[h].cpu().numpy() - exact.sum(axis=0)) <= v["bound"])
        assert_attn_bound(a.bound[h].cpu().numpy(), v["bound"], np.abs(oracle.bf16_to_f64(dOb)).sum(axis=0))
