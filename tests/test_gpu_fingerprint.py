"""GPU fingerprint and xorsum parity with the oracle, element for element.

Sizes span several chunks with ragged tails, unaligned starts, every element
width, empty tensors and the tiny workload.  The bar is bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import sdc_workloads as W
from tests._helpers import fp_table, host_bits, oracle_fp_table

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _random_tensor(numel, dtype, gen):
    if dtype.is_floating_point:
        return W.normal((numel,), 0.02, dtype, gen, DEV)
    info = torch.iinfo(dtype)
    return torch.randint(info.min, info.max, (numel,), generator=gen, device=DEV, dtype=torch.int64).to(dtype)


def test_tiny_workload(sdc):
    w = W.tiny(DEV, seed=0)
    plan = sdc.Plan(w["replicas"])
    got = fp_table(plan.fingerprint())
    ref = oracle_fp_table(w["replicas"])
    assert got == ref
    t = w["truth"]
    assert got[1][t["tensor"]] != got[0][t["tensor"]]
    assert got[0] == got[2]


@pytest.mark.parametrize("dtype", [torch.uint8, torch.int16, torch.bfloat16, torch.float16, torch.float32,
                                   torch.int32, torch.float64, torch.int64])
@pytest.mark.parametrize("chunk_bytes", [4096, 16384, 32768])
def test_sizes_and_offsets(sdc, dtype, chunk_bytes):
    """Tensors of ragged sizes at unaligned element offsets inside one buffer."""
    gen = W.generator(11, DEV)
    es = torch.empty(0, dtype=dtype).element_size()
    sizes = [0, 1, 2, 3, 7, 15, 16, 17, 31, 100, 1000, 4097, 65537, 3 * chunk_bytes // es + 5, 200_001]
    total = sum(sizes) + 64 * len(sizes)
    flat = _random_tensor(total, dtype, gen)
    tensors, off = [], 1  # start one element past an aligned boundary
    for i, n in enumerate(sizes):
        tensors.append(flat[off: off + n])
        off += n + (i % 5) + 1
    reps = [tensors, [t.clone() for t in tensors]]
    plan = sdc.Plan(reps, chunk_bytes=chunk_bytes)
    got = fp_table(plan.fingerprint())
    assert got == oracle_fp_table(reps)


def test_maximum_chunk_fill_16bit_extremes(sdc):
    """All-(-32768) and all-32767 int16 chunks: the 32-bit in-chunk sums at their bounds."""
    for v in (-32768, 32767, -1):
        t = torch.full((3 * 16384 + 11,), v, dtype=torch.int16, device=DEV)
        plan = sdc.Plan([[t]], chunk_bytes=32768)
        assert fp_table(plan.fingerprint()) == oracle_fp_table([[t]])
    t = torch.full((3 * 32768 + 7,), 255, dtype=torch.uint8, device=DEV)
    plan = sdc.Plan([[t]], chunk_bytes=32768)
    assert fp_table(plan.fingerprint()) == oracle_fp_table([[t]])
    t = torch.full((9 * 8192 + 3,), -(2 ** 31), dtype=torch.int32, device=DEV)
    plan = sdc.Plan([[t]], chunk_bytes=32768)
    assert fp_table(plan.fingerprint()) == oracle_fp_table([[t]])


def test_mixed_dtypes_many_replicas(sdc):
    gen = W.generator(12, DEV)
    base = [_random_tensor(n, dt, gen) for n, dt in
            [(5000, torch.float32), (777, torch.bfloat16), (12345, torch.float16), (99, torch.uint8),
             (0, torch.float32), (31, torch.float64)]]
    R = 7
    reps = [[t.clone() for t in base] for _ in range(R)]
    W.xor_element(reps[3][0], 4321, 1 << 22)
    W.xor_element(reps[5][2], 0, 1 << 15)
    plan = sdc.Plan(reps)
    got = fp_table(plan.fingerprint())
    assert got == oracle_fp_table(reps)


def test_pages_weight_faults_detected(sdc):
    """Bit flip, swap and +-4096 compensating change (the page's weight faults)."""
    gen = W.generator(13, DEV)
    w = W.normal((4096, 256), 0.02, torch.float32, gen, DEV)
    reps = [[w.clone()] for _ in range(3)]
    plan = sdc.Plan(reps)
    base = fp_table(plan.fingerprint())[0][0]
    x = reps[1][0].view(-1)
    bits = x.view(torch.int32)
    # bit 22 flip
    bits[100] ^= 1 << 22
    got = fp_table(plan.fingerprint())
    assert got[1][0][0] != base[0] and got[0][0] == base
    bits[100] ^= 1 << 22
    # swap two values: plain sum unchanged, weighted sum differs
    a, b = x[10].clone(), x[20].clone()
    x[10], x[20] = b, a
    got = fp_table(plan.fingerprint())
    assert got[1][0][0] == base[0] and got[1][0][1] != base[1]
    x[10], x[20] = a, b
    # +4096 / -4096 on two bit patterns
    bits[10] += 4096
    bits[20] -= 4096
    got = fp_table(plan.fingerprint())
    assert got[1][0][0] == base[0] and got[1][0][1] != base[1]
    assert got == oracle_fp_table(reps)


def test_repeatable_and_independent_of_launch_shape(sdc):
    gen = W.generator(14, DEV)
    reps = [[W.normal((1 << 20,), 0.02, torch.float32, gen, DEV), W.normal((333,), 0.02, torch.bfloat16, gen, DEV)]]
    outs = []
    for cb, ctas in [(16384, 0), (4096, 1), (32768, 2)]:
        plan = sdc.Plan(reps, chunk_bytes=cb, ctas_per_sm=ctas)
        outs.append(fp_table(plan.fingerprint()))
        outs.append(fp_table(plan.fingerprint()))
    assert all(o == outs[0] for o in outs)


def test_xorsum_parity(sdc):
    gen = W.generator(15, DEV)
    base = [_random_tensor(n, dt, gen) for n, dt in
            [(10001, torch.float32), (7, torch.uint8), (65536 + 3, torch.bfloat16), (0, torch.float16),
             (4099, torch.float64), (5, torch.int16)]]
    reps = [base, [t.clone() for t in base]]
    W.xor_element(reps[1][2], 5000, 1 << 9)
    plan = sdc.Plan(reps)
    got = plan.xorsum().cpu().numpy().view(np.uint64)
    for r in range(2):
        for k, t in enumerate(reps[r]):
            assert int(got[r, k]) == oracle.xorsum(host_bits(t)), (r, k)
    mism, diff = sdc.xorsum_compare(plan.xorsum()[0], plan.xorsum()[1])
    assert mism.cpu().tolist() == [0, 0, 1, 0, 0, 0]
    assert int(diff.cpu().numpy().view(np.uint64)[2]) == 1 << 9


def test_errors_on_device(sdc):
    t = torch.zeros(100, dtype=torch.float32, device=DEV)
    with pytest.raises(sdc.SdcError) as ei:  # host memory
        h = torch.zeros(100, dtype=torch.float32)
        d = np.zeros(1, dtype=sdc.DESC_DTYPE)
        d[0] = (h.data_ptr(), 100, 4, 1)
        sdc.sdc_plan_create(d, 1, 1)
    assert ei.value.status == 8
    d = np.zeros(1, dtype=sdc.DESC_DTYPE)
    d[0] = (t.data_ptr(), 10 ** 9, 4, 1)  # runs past its allocation
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_plan_create(d, 1, 1)
    assert ei.value.status == 8
    plan = sdc.Plan([[t]])
    out = torch.empty((1, 1, 2), dtype=torch.int64, device=DEV)
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_fingerprint(plan.handle, out.data_ptr(), plan.ws.data_ptr(), 8, 0)
    assert ei.value.status == 5
    raw = sdc.Plan([[torch.zeros(10, dtype=torch.uint8, device=DEV)]])
    with pytest.raises(sdc.SdcError) as ei:
        raw.grad_scan()
    assert ei.value.status == 7
