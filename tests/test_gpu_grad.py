"""GPU gradient scans versus the oracle: non-finite counts exactly, the squared
norm within 1e-10 relative, the average bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import host_bits, stats_match

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _specials(t: torch.Tensor, gen_seed: int, n: int):
    """Plant NaN/Inf/huge/tiny/zero values at seeded positions (ground truth returned)."""
    rng = np.random.default_rng(gen_seed)
    vals = [float("nan"), float("inf"), float("-inf"), 2.0 ** 70, -(2.0 ** 70), 0.0, -0.0, 1e-40, 40.0, -1e30]
    flat = t.view(-1)
    pos = rng.choice(flat.numel(), size=min(n, flat.numel()), replace=False)
    for p in pos:
        v = vals[int(rng.integers(len(vals)))]
        flat[int(p)] = torch.tensor(v, dtype=torch.float32).to(t.dtype)
    return pos


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("n_bufs", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("numel", [0, 1, 7, 8193, 3 * 8192 + 5, 100_003])
def test_average_scan_parity(sdc, dtype, n_bufs, numel):
    gen = W.generator(numel + n_bufs, DEV)
    std = 1e-3 if dtype != torch.float16 else 1e-2
    bufs = [W.normal((numel,), std, dtype, gen, DEV) for _ in range(n_bufs)]
    if numel > 50:
        _specials(bufs[0], numel, 12)
    avg, pre, post = sdc.grad_average_scan(bufs)
    torch.cuda.synchronize()
    name = NAMES[dtype]
    hb = [host_bits(b) for b in bufs]
    ref_avg = oracle.average(hb, name)
    assert np.array_equal(host_bits(avg), ref_avg)
    got_pre = sdc.decode_stats(pre)
    for b in range(n_bufs):
        stats_match(got_pre[b], oracle.grad_stats(hb[b], name))
    stats_match(sdc.decode_stats(post)[0], oracle.grad_stats(ref_avg, name))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_average_scan_unaligned_element_path(sdc, dtype):
    gen = W.generator(21, DEV)
    big = [W.normal((50_001,), 1e-3, dtype, gen, DEV) for _ in range(4)]
    bufs = [b[1:] for b in big]  # start one element past a 16-byte boundary
    _specials(bufs[2], 5, 20)
    avg, pre, post = sdc.grad_average_scan(bufs)
    hb = [host_bits(b) for b in bufs]
    ref_avg = oracle.average(hb, NAMES[dtype])
    assert np.array_equal(host_bits(avg), ref_avg)
    for b in range(4):
        stats_match(sdc.decode_stats(pre)[b], oracle.grad_stats(hb[b], NAMES[dtype]))
    stats_match(sdc.decode_stats(post)[0], oracle.grad_stats(ref_avg, NAMES[dtype]))


def test_edge_values_bf16(sdc):
    # subnormals, the |x| >= 32 slow path, 2^64 (first big), largest finite, signed zeros
    vals = np.array([0x0001, 0x807F, 0x4200, 0x5F7F, 0x5F80, 0x7F7F, 0xFF7F, 0x0000, 0x8000, 0x3F80] * 1000,
                    dtype=np.uint16)
    t = torch.from_numpy(vals.view(np.int16)).to(DEV).view(torch.bfloat16)
    avg, pre, post = sdc.grad_average_scan([t, t.clone(), t.clone(), t.clone()])
    ref = oracle.grad_stats(vals, "bf16")
    got = sdc.decode_stats(pre)[0]
    stats_match(got, ref)
    assert got["n_big"] == 3000  # 2^64, bf16 max, -bf16 max
    assert np.array_equal(host_bits(avg), oracle.average([vals] * 4, "bf16"))


def test_edge_values_f32(sdc):
    f = np.array([1e-45, -3e-39, 2.0 ** -60, 2.0 ** -52, 1.0, 1.8e19, 1.9e19, 3e38, 0.0, -0.0], dtype=np.float32)
    t = torch.from_numpy(np.tile(f, 777)).to(DEV)
    avg, pre, post = sdc.grad_average_scan([t])
    stats_match(sdc.decode_stats(pre)[0], oracle.grad_stats(np.tile(f, 777), "f32"))
    assert np.array_equal(host_bits(avg), host_bits(t))


def test_nan_propagation_and_canonical_output(sdc):
    a = torch.zeros(4096, dtype=torch.bfloat16, device=DEV)
    b = a.clone()
    a[5] = float("inf")
    b[5] = float("-inf")
    a[9] = float("nan")
    a.view(torch.int16)[11] = 0x7F81  # NaN with a payload
    avg, pre, post = sdc.grad_average_scan([a, b])
    bits = host_bits(avg)
    assert bits[5] == 0x7FC0 and bits[9] == 0x7FC0 and bits[11] == 0x7FC0
    post_s = sdc.decode_stats(post)[0]
    assert post_s["n_nan"] == 3 and math.isnan(post_s["norm"]) and post_s["nonfinite_fp32"] == 1


def test_plan_grad_scan_parity(sdc):
    gen = W.generator(22, DEV)
    layout = [((3000,), torch.bfloat16), ((77, 13), torch.float32), ((9,), torch.float16), ((0,), torch.float32),
              ((65536 + 1,), torch.bfloat16)]
    reps = []
    for r in range(3):
        ts = [W.normal(s, 1e-3, dt, gen, DEV) for s, dt in layout]
        reps.append(ts)
    _specials(reps[1][0], 1, 30)
    _specials(reps[2][4], 2, 50)
    # unaligned copies of the same data in replica 2's second tensor
    flat = torch.empty(77 * 13 + 1, dtype=torch.float32, device=DEV)
    flat[1:].copy_(reps[2][1].view(-1))
    reps[2][1] = flat[1:].view(77, 13)
    plan = sdc.Plan(reps)
    got = sdc.decode_stats(plan.grad_scan())
    for r in range(3):
        ref = oracle.grad_stats_multi([host_bits(t) for t in reps[r]], [NAMES[t.dtype] for t in reps[r]])
        stats_match(got[r], ref)


def test_repeatable(sdc):
    g = W.grads_flat(1_000_003, 4, torch.bfloat16, 1e-3, DEV, seed=7, rate=1e-5)
    ws = torch.empty(1 << 24, dtype=torch.uint8, device=DEV)
    results = []
    for _ in range(3):
        avg, pre, post = sdc.grad_average_scan(g["bufs"], ws=ws)
        results.append((host_bits(avg).tobytes(), pre.cpu().numpy().tobytes(), post.cpu().numpy().tobytes()))
    assert results[0] == results[1] == results[2]


@pytest.mark.parametrize("dtype,magnitudes", [
    (torch.bfloat16, (3.0, 3.0)),     # after the 2^118 scaling each packed half of a run stays finite,
    (torch.bfloat16, (2.85, 3.98)),   # but the two halves' sum overflows float32
    (torch.float32, (1.35e19, 1.35e19)),  # x^2 finite, two of them past FLT_MAX: the norm alarm
])
def test_run_halves_whose_sum_overflows(sdc, dtype, magnitudes):
    gen = torch.Generator(device="cpu").manual_seed(41)
    n = 3 * 8192 + 5
    lo, hi = magnitudes
    mag = lo + (hi - lo) * torch.rand(n, generator=gen, dtype=torch.float64)
    sign = torch.where(torch.rand(n, generator=gen) < 0.5, -1.0, 1.0).to(torch.float64)
    bufs = [(mag * sign).to(dtype).to(DEV) for _ in range(2)]
    name = NAMES[dtype]
    hb = [host_bits(b) for b in bufs]
    ref = oracle.grad_stats(hb[0], name)
    assert math.isfinite(ref["sumsq_finite"])
    avg, pre, post = sdc.grad_average_scan(bufs)
    for b in range(2):
        stats_match(sdc.decode_stats(pre)[b], oracle.grad_stats(hb[b], name))
    stats_match(sdc.decode_stats(post)[0], oracle.grad_stats(host_bits(avg), name))
    plan = sdc.Plan([[bufs[0]], [bufs[1]]])
    got = sdc.decode_stats(plan.grad_scan())
    for b in range(2):
        stats_match(got[b], oracle.grad_stats(hb[b], name))


def _block_pattern(kind: str, n: int, dtype, seed: int) -> torch.Tensor:
    """Magnitude patterns in blocks of 2,048 elements (one 8-vector run of every lane of a
    warp task) that defeat an offset taken from the previous run: jumps by 2^20 both ways,
    steady growth, zero blocks, squares below float32's range, sums past FLT_MAX,
    single spikes inside a run and subnormals."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n, generator=gen, dtype=torch.float64)
    blk = torch.arange(n) // 2048
    f16 = dtype == torch.float16
    if kind == "alternate":
        scale = torch.where(blk % 2 == 0, 1.0, 2.0 ** (-12 if f16 else -20)).to(torch.float64)
    elif kind == "grow":
        scale = torch.pow(torch.tensor(2.0, dtype=torch.float64), (blk % 8).to(torch.float64) * (1 if f16 else 3))
        scale = scale * (2.0 ** -8 if f16 else 1.0)
    elif kind == "zero_blocks":
        scale = torch.where(blk % 3 == 1, 0.0, 1e-3).to(torch.float64)
    elif kind == "tiny":
        scale = torch.where(blk % 2 == 0, 2.0 ** (-20 if f16 else -70), 1e-3).to(torch.float64)
    elif kind == "near_overflow":
        scale = torch.full((n,), 2.0 ** (10 if f16 else 62), dtype=torch.float64)
    elif kind == "spikes":
        scale = torch.full((n,), 1e-3, dtype=torch.float64)
        idx = torch.arange(5, n, 997)
        scale[idx] = 1e-3 * 2.0 ** (8 if f16 else 16)
    elif kind == "subnormal":
        scale = torch.full((n,), 2.0 ** (-20 if f16 else -130), dtype=torch.float64)
    else:
        raise ValueError(kind)
    return (x * scale).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind", ["alternate", "grow", "zero_blocks", "tiny", "near_overflow", "spikes",
                                  "subnormal"])
def test_offset_runs_adversarial(sdc, dtype, kind):
    # the 16-bit scans start each run's sum at an offset from the previous run; runs whose
    # magnitudes break that guess must be redone (or summed exactly), never accepted inexactly
    n = 4 * 8192 + 5
    bufs = [_block_pattern(kind, n, dtype, 60 + i).to(DEV) for i in range(2)]
    bufs.append(torch.flip(bufs[0], dims=[0]).contiguous())
    name = NAMES[dtype]
    hb = [host_bits(b) for b in bufs]
    avg, pre, post = sdc.grad_average_scan(bufs)
    ref_avg = oracle.average(hb, name)
    assert np.array_equal(host_bits(avg), ref_avg)
    got = sdc.decode_stats(pre)
    for b in range(3):
        stats_match(got[b], oracle.grad_stats(hb[b], name))
    stats_match(sdc.decode_stats(post)[0], oracle.grad_stats(ref_avg, name))
    plan = sdc.Plan([[b] for b in bufs])
    got = sdc.decode_stats(plan.grad_scan())
    for b in range(3):
        stats_match(got[b], oracle.grad_stats(hb[b], name))
