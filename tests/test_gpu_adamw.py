"""GPU clip + AdamW step + fingerprint of the written weights versus the oracle,
bit for bit, including the device-side gate and the page's optimizer-step fault."""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import fp_table, host_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
HP = {"lr": 3e-4, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1, "max_grad_norm": 1.0}
NAMES = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _setup(R, sizes, gdtype, seed, misalign_moments=False):
    gen = W.generator(seed, DEV)
    base = [W.normal((n,), 0.02, torch.float32, gen, DEV) for n in sizes]
    weights = [[t.clone() for t in base] for _ in range(R)]
    grads = [W.normal((n,), 1e-2, gdtype, gen, DEV) for n in sizes]

    def moment(n, positive):
        t = W.normal((n + 1,), 1e-3, torch.float32, gen, DEV)
        if positive:
            t = t.abs() * 1e-3
        return t[1:] if misalign_moments else t[:n]

    m0 = [moment(n, False) for n in sizes]
    v0 = [moment(n, True) for n in sizes]
    # data-parallel replicas hold identical optimizer states (copies keep the views' alignment)
    m = [m0] + [[_same_alignment_copy(t) for t in m0] for _ in range(R - 1)]
    v = [v0] + [[_same_alignment_copy(t) for t in v0] for _ in range(R - 1)]
    return weights, grads, m, v


def _same_alignment_copy(t):
    off = (t.data_ptr() % 16) // 4
    buf = torch.empty(t.numel() + off, dtype=t.dtype, device=t.device)
    out = buf[off:]
    out.copy_(t)
    return out


def _oracle_step(weights, grads, m, v, hp, post):
    """The oracle applied to host copies; returns (weights, m, v) as float32 arrays."""
    R, T = len(weights), len(grads)
    ow = [[host_bits(t).view(np.float32).copy() for t in ws] for ws in weights]
    om = [[host_bits(t).view(np.float32).copy() for t in ms] for ms in m]
    ov = [[host_bits(t).view(np.float32).copy() for t in vs] for vs in v]
    for r in range(R):
        for k in range(T):
            oracle.adamw_step(ow[r][k], host_bits(grads[k]), NAMES[grads[k].dtype], om[r][k], ov[r][k], hp, post)
    return ow, om, ov


def _assert_state(weights, m, v, ow, om, ov):
    for r in range(len(weights)):
        for k in range(len(weights[0])):
            assert np.array_equal(host_bits(weights[r][k]), ow[r][k].view(np.uint32)), (r, k)
            assert np.array_equal(host_bits(m[r][k]), om[r][k].view(np.uint32)), (r, k)
            assert np.array_equal(host_bits(v[r][k]), ov[r][k].view(np.uint32)), (r, k)


@pytest.mark.parametrize("gdtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("misalign", [False, True])
def test_step_parity_no_clip(sdc, gdtype, misalign):
    sizes = [1, 3, 4, 5, 17, 1000, 4097, 3 * 4096 + 7, 65537]
    weights, grads, m, v = _setup(2, sizes, gdtype, seed=len(sizes) + int(misalign), misalign_moments=misalign)
    plan = sdc.Plan(weights)
    opt = sdc.AdamWFingerprint(plan, grads, m, v)
    for step in (1, 2, 3):
        hp = dict(HP, step=step, clip=0)
        ow, om, ov = _oracle_step(weights, grads, m, v, hp, None)
        fp = opt.step(hp)
        torch.cuda.synchronize()
        _assert_state(weights, m, v, ow, om, ov)
        ref = [[oracle.fingerprint(ow[r][k].view(np.uint32)) for k in range(len(sizes))] for r in range(2)]
        assert fp_table(fp) == ref
        assert fp_table(fp) == fp_table(plan.fingerprint())  # fused == re-read of the stored weights


def test_clip_and_gate_from_device_stats(sdc):
    sizes = [4096, 333, 70_001]
    weights, grads32, m, v = _setup(3, sizes, torch.float32, seed=9)
    # the averaged gradient and its stats from the fused average-scan (4 local buffers, float32)
    local = [[(g * (1.0 + 0.1 * b)).contiguous() for g in grads32] for b in range(4)]
    flat_local = [torch.cat(ls) for ls in local]
    avg, pre, post = sdc.grad_average_scan(flat_local)
    grads = list(torch.split(avg, sizes))
    post_d = sdc.decode_stats(post)[0]
    ref_avg = oracle.average([host_bits(b) for b in flat_local], "f32")
    ref_post = oracle.grad_stats(ref_avg, "f32")
    assert ref_post["norm"] > 1.0  # the clip coefficient is below 1
    plan = sdc.Plan(weights)
    opt = sdc.AdamWFingerprint(plan, grads, m, v)
    hp = dict(HP, step=1, clip=1)
    ow, om, ov = _oracle_step(weights, grads, m, v, hp, ref_post)
    fp = opt.step(hp, post=post)
    torch.cuda.synchronize()
    _assert_state(weights, m, v, ow, om, ov)
    assert fp_table(fp) == fp_table(plan.fingerprint())
    # a non-finite reduced gradient: the step is skipped on the device
    bad = post.clone()
    raw = np.frombuffer(bad.cpu().numpy().tobytes(), dtype=sdc.GRAD_STATS_DTYPE).copy()
    raw["nonfinite_fp32"] = 1
    raw["norm"] = float("nan")
    bad.copy_(torch.from_numpy(raw.view(np.uint8)))
    before = [[host_bits(t).copy() for t in ws] for ws in weights]
    fp2 = opt.step(dict(HP, step=2, clip=1), post=bad)
    torch.cuda.synchronize()
    for r in range(3):
        for k in range(len(sizes)):
            assert np.array_equal(host_bits(weights[r][k]), before[r][k])
    assert fp_table(fp2) == fp_table(fp)


def test_optimizer_state_fault_is_named_by_the_vote(sdc):
    """The page's optimizer-step fault: one replica's update goes wrong (here a bit
    of its exp_avg); its fingerprints differ after the fused step and the vote
    names it."""
    sizes = [2048, 511, 9000]
    weights, grads, m, v = _setup(3, sizes, torch.bfloat16, seed=11)
    W.xor_element(m[2][1], 17, 1 << 20)
    plan = sdc.Plan(weights)
    opt = sdc.AdamWFingerprint(plan, grads, m, v)
    fp = opt.step(dict(HP, step=1, clip=0))
    suspect, mask, summary = sdc.vote(fp)
    assert suspect.cpu().tolist() == [-1, 2, -1]
    assert sdc.pages_verdict(sdc.decode_summary(summary)) == {"diverged": True, "suspects": [2]}
