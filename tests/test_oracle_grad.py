"""Pins of the oracle's gradient statistics and average.

Sources: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" -- "Step 1: Detect" (worked example), "Check 1: NaN/Inf
gradients, before and after the all-reduce", "Decide what the alarm means".
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f16_bits(x: np.ndarray) -> np.ndarray:
    return x.astype(np.float16).view(np.uint16)


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [0, 1, 9, 1000])
def test_sumsq_equals_fsum(dtype, n):
    # math.fsum is the correctly rounded sum of the (exact) float64 squares
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n) * 10.0 ** rng.integers(-30, 10, size=n)
    if dtype == "f32":
        raw = x.astype(np.float32)
        vals = raw.astype(np.float64)
    elif dtype == "bf16":
        raw = _bf16_bits(x)
        vals = _bf16_values(raw)
    else:
        raw = _f16_bits(np.clip(x, -6e4, 6e4))
        vals = raw.view(np.float16).astype(np.float64)
    st = oracle.grad_stats(raw, dtype)
    assert st["sumsq_finite"] == math.fsum(v * v for v in vals)
    assert st["n_nan"] == st["n_inf"] == 0
    assert st["n_elems"] == n


def test_closed_form_constant():
    # n copies of c: sum of squares is exactly n * c^2 when that is representable
    c = np.float32(0.375)
    st = oracle.grad_stats(np.full(1 << 20, c, dtype=np.float32), "f32")
    assert st["sumsq_finite"] == (1 << 20) * 0.375 ** 2
    assert st["norm"] == math.sqrt((1 << 20) * 0.375 ** 2)


def test_subnormals_exact():
    tiny = np.array([1, 3, 0x7F], dtype=np.uint16)  # bf16 subnormals
    st = oracle.grad_stats(tiny, "bf16")
    assert st["sumsq_finite"] == math.fsum([(k * 2.0 ** -133) ** 2 for k in (1, 3, 127)])
    f32 = np.array([1, 2], dtype=np.uint32).view(np.float32)  # f32 subnormals 2^-149, 2^-148
    assert oracle.grad_stats(f32, "f32")["sumsq_finite"] == 2.0 ** -298 + 2.0 ** -296


def test_injected_counts_ground_truth():
    rng = np.random.default_rng(1)
    n = 200_000
    x = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    bits = _bf16_bits(x)
    pos = rng.choice(n, size=40, replace=False)
    kinds = rng.integers(0, 5, size=40)
    table = {0: 0x7FC0, 1: 0x7F80, 2: 0xFF80, 3: 0x6300, 4: 0xE300}  # NaN, +Inf, -Inf, +2^70, -2^70
    for p, k in zip(pos, kinds):
        bits[p] = table[int(k)]
    st = oracle.grad_stats(bits, "bf16")
    assert st["n_nan"] == int((kinds == 0).sum())
    assert st["n_inf"] == int(((kinds == 1) | (kinds == 2)).sum())
    assert st["n_big"] == int(((kinds == 3) | (kinds == 4)).sum())
    assert math.isnan(st["norm"]) == bool((kinds == 0).any())
    assert st["nonfinite_fp32"] == 1


def test_norm_ieee_propagation():
    st = oracle.grad_stats(np.array([1.0, np.inf, 2.0], dtype=np.float32), "f32")
    assert st["norm"] == math.inf and st["n_inf"] == 1 and st["sumsq_finite"] == 5.0
    st = oracle.grad_stats(np.array([np.nan, np.inf], dtype=np.float32), "f32")
    assert math.isnan(st["norm"])


def test_overflow_threshold_page_value():
    g = json.load(open(os.path.join(GOLDEN, "alarm_thresholds.json")))
    thr = math.sqrt(oracle.FLT_MAX)
    assert abs(thr - g["printed_threshold_approx"]) / g["printed_threshold_approx"] < 0.03
    # bf16: 2^64 is the first value whose square overflows float32
    below = np.array([0x5F7F], dtype=np.uint16)  # (2 - 2^-7) * 2^63
    at = np.array([0x5F80], dtype=np.uint16)     # 2^64
    assert oracle.grad_stats(below, "bf16")["n_big"] == 0
    assert oracle.grad_stats(below, "bf16")["nonfinite_fp32"] == 0
    assert oracle.grad_stats(at, "bf16")["n_big"] == 1
    assert oracle.grad_stats(at, "bf16")["nonfinite_fp32"] == 1
    # f32 neighbours of sqrt(FLT_MAX)
    f = np.array([np.nextafter(np.float32(2.0 ** 64), np.float32(0)), np.float32(2.0 ** 64)], dtype=np.float32)
    assert oracle.grad_stats(f[:1], "f32")["n_big"] == 0
    assert oracle.grad_stats(f[1:], "f32")["n_big"] == 1
    # many moderate values whose squares sum past FLT_MAX also raise the float32 flag
    many = np.full(4, np.float32(1.2e19), dtype=np.float32)
    st = oracle.grad_stats(many, "f32")
    assert st["n_big"] == 0 and st["nonfinite_fp32"] == 1 and math.isfinite(st["norm"])
    # float16 squares never overflow float32
    assert oracle.grad_stats(_f16_bits(np.array([65504.0])), "f16")["n_big"] == 0


# ---------------------------------------------------------------- rounding + average
def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    # ties, subnormals, near-overflow values
    special = np.array([0x3F808000, 0x3F818000, 0x00008000, 0x00018000, 0x7F7F8000, 0x7F7FFFFF,
                        0x80000001, 0x007FFFFF, 0x7F800000, 0xFF800000, 0x3F7FFFFF], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    vals = bits.view(np.float32)
    vals = vals[~np.isnan(vals)]
    ref = torch.from_numpy(vals.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.round_f32(float(v), "bf16") for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.round_f32(float("nan"), "bf16") == 0x7FC0


def test_round_to_f16_matches_numpy():
    rng = np.random.default_rng(3)
    vals = (rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, size=20000)).astype(np.float32)
    vals = np.concatenate([vals, np.array([65519.0, 65520.0, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -24 * 1.5],
                                          dtype=np.float32)])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.round_f32(float(v), "f16") for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_worked_example_average_and_update():
    g = json.load(open(os.path.join(GOLDEN, "ddp_worked_example.json")))
    lr = np.float32(g["learning_rate"])
    w0 = np.float32(g["weight_at_start"])

    def step(grads):
        bufs = [np.array([v], dtype=np.float32) for v in grads]
        avg = oracle.average(bufs, "f32").view(np.float32)[0]
        weights = [np.float32(w0 - lr * avg) for _ in grads]  # every replica applies the same average
        return avg, weights

    avg, weights = step(g["local_gradients"])
    assert round(float(avg), 2) == g["averaged_gradient_printed"]
    assert round(float(weights[0]), 3) == g["weight_after_step_printed"]
    fps = [oracle.fingerprint(np.array([w], dtype=np.float32)) for w in weights]
    assert len(set(fps)) == 1
    suspect, mask, summ = oracle.vote([[fp] for fp in fps])
    assert oracle.pages_verdict(summ) == {"diverged": False, "suspects": []}

    faulty = list(g["local_gradients"])
    faulty[g["fault"]["replica"]] = g["fault"]["local_gradient"]
    avg_f, weights_f = step(faulty)
    fps_f = [oracle.fingerprint(np.array([w], dtype=np.float32)) for w in weights_f]
    assert len(set(fps_f)) == 1  # the fault reached every replica alike
    assert oracle.pages_verdict(oracle.vote([[fp] for fp in fps_f])[2])["diverged"] is False
    assert round(float(weights_f[0]), 3) == 0.350  # derived, not printed
    # the fault is visible only in the faulty replica's local gradient, before averaging
    pre = [oracle.fingerprint(np.array([v], dtype=np.float32)) for v in faulty]
    assert pre[1] != pre[0] and pre[1] != pre[2]


def test_average_closed_forms():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(5000) * 1e-3).astype(np.float32)
    b = _bf16_bits(x)
    # four identical buffers average to themselves
    assert np.array_equal(oracle.average([b, b, b, b], "bf16"), b)
    # NaN in one input gives the canonical NaN; +Inf and -Inf give NaN; Inf alone stays Inf
    nan_in = b.copy(); nan_in[3] = 0xFFC1
    pinf = b.copy(); pinf[4] = 0x7F80
    ninf = b.copy(); ninf[4] = 0xFF80
    out = oracle.average([nan_in, b, pinf, b], "bf16")
    assert out[3] == 0x7FC0 and out[4] == 0x7F80
    out = oracle.average([pinf, ninf, b, b], "bf16")
    assert out[4] == 0x7FC0
    # a float32 average rounded by torch's conversion
    bufs = [_bf16_bits(rng.standard_normal(5000).astype(np.float32)) for _ in range(4)]
    acc = _bf16_values(bufs[0]).astype(np.float32)
    for bb in bufs[1:]:
        acc = (acc + _bf16_values(bb).astype(np.float32)).astype(np.float32)
    acc = (acc * np.float32(0.25)).astype(np.float32)
    assert np.array_equal(oracle.average(bufs, "bf16"), _bf16_bits(acc))


def test_closed_form_magnitudes_three_to_four():
    # n copies of c with |c| between 3 and 4 (exact in bf16): the sum of squares is exactly n c^2,
    # nothing is big and no float32 alarm is raised
    for c in (3.0, -3.5, 3.984375):
        st = oracle.grad_stats(_bf16_bits(np.full(4099, c)), "bf16")
        assert st["sumsq_finite"] == 4099 * c * c
        assert st["n_big"] == 0 and st["nonfinite_fp32"] == 0
