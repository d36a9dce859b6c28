"""Pins of the oracle's clipped AdamW step.

Source: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" -- "Use case: Testing the checks on SageMaker HyperPod"
(AdamW, betas (0.9, 0.95), weight decay 0.1, clipping at 1.0) and `train()`
(clip, reduced-gradient gate, step).
"""
import math

import numpy as np
import pytest
import torch

import oracle

HP = {"lr": 3e-4, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1, "max_grad_norm": 1.0, "clip": 1}


@pytest.mark.parametrize("steps", [1, 3, 10])
def test_matches_torch_adamw(steps):
    # torch's own AdamW (single-tensor path) on CPU is a separate implementation of the
    # same update (it rounds some steps differently, e.g. a fused multiply-add in its
    # lerp); agreement to float32 rounding of the update -- absolute 1e-9 on weights
    # moved by ~3e-4 per step -- pins every term, sign and operand: a dropped weight
    # decay alone would differ by ~6e-7
    rng = np.random.default_rng(steps)
    n = 10_000
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    param = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([param], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"], foreach=False)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, steps + 1):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        param.grad = torch.from_numpy(g.copy())
        opt.step()
        oracle.adamw_step(p, g, "f32", m, v, dict(HP, step=t, clip=0), None)
    st = opt.state[param]
    np.testing.assert_allclose(p, param.detach().numpy(), rtol=1e-6, atol=1e-9)
    # the moments cancel near zero too: absolute tolerance a few float32 ulps of their scale
    for mine, ref in ((m, st["exp_avg"].numpy()), (v, st["exp_avg_sq"].numpy())):
        np.testing.assert_allclose(mine, ref, rtol=1e-6, atol=2e-6 * float(np.abs(ref).max()))


def test_clip_coefficient_matches_torch_clip_grad_norm():
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(4096) * 0.5).astype(np.float32)
    t = torch.from_numpy(g.copy()).requires_grad_(False)
    param = torch.nn.Parameter(torch.zeros(4096))
    param.grad = t.clone()
    total = torch.nn.utils.clip_grad_norm_([param], 1.0)
    st = oracle.grad_stats(g, "f32")
    assert abs(st["norm"] - float(total)) <= 1e-6 * st["norm"]
    coef = oracle.clip_coef(st["norm"], 1.0)
    np.testing.assert_allclose(param.grad.numpy(), g * np.float32(coef), rtol=2e-7)


def test_closed_forms():
    n = 64
    p = np.full(n, 0.5, np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    # zero gradient: only the decoupled weight decay acts
    oracle.adamw_step(p, np.zeros(n, np.float32), "f32", m, v, dict(HP, step=1, clip=0), None)
    assert np.all(p == np.float32(np.float32(0.5) * np.float32(1 - np.float32(3e-4) * np.float32(0.1))))
    assert np.all(m == 0) and np.all(v == 0)
    # first step with a constant gradient: bias-corrected moments give ~lr * sign(g)
    p = np.zeros(n, np.float32)
    oracle.adamw_step(p, np.full(n, -0.25, np.float32), "f32", m, v, dict(HP, step=1, clip=0, weight_decay=0.0), None)
    assert np.allclose(p, 3e-4, rtol=1e-5)


def test_gate_skips_the_step_on_the_reduced_gradient_alarm():
    p = np.ones(8, np.float32)
    m = np.zeros(8, np.float32)
    v = np.zeros(8, np.float32)
    bad = {"nonfinite_fp32": 1, "norm": math.nan}
    assert oracle.adamw_step(p, np.ones(8, np.float32), "f32", m, v, dict(HP, step=1), bad) is False
    assert np.all(p == 1) and np.all(m == 0) and np.all(v == 0)


def test_bf16_gradients_are_read_exactly():
    g32 = np.array([1.5, -2.25, 3e-5], np.float32)
    gbf = torch.from_numpy(g32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    back = torch.from_numpy(gbf.view(np.int16)).view(torch.bfloat16).float().numpy()
    p1, m1, v1 = np.zeros(3, np.float32), np.zeros(3, np.float32), np.zeros(3, np.float32)
    p2, m2, v2 = p1.copy(), m1.copy(), v1.copy()
    oracle.adamw_step(p1, gbf, "bf16", m1, v1, dict(HP, step=2, clip=0), None)
    oracle.adamw_step(p2, back, "f32", m2, v2, dict(HP, step=2, clip=0), None)
    assert np.array_equal(p1, p2) and np.array_equal(m1, m2) and np.array_equal(v1, v2)
