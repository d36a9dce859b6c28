"""Pins of the oracle's fingerprint and xorsum against facts fixed outside it.

Fingerprint definition: "Detecting and recovering from silent data corruption
on Amazon SageMaker HyperPod", section "Compare by fingerprint".  Xorsum:
"Safeguarding LLM Training at Scale ..." review, method section 4.
"""
import json
import os
from functools import reduce

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1
VIEWS = {1: np.uint8, 2: np.int16, 4: np.int32, 8: np.int64}


def _brute_fp(raw: bytes, esize: int):
    """Python big-int brute force: bytes -> ints of the page's bit view -> sums mod 2^64."""
    signed = esize != 1
    s = w = 0
    for i in range(len(raw) // esize):
        b = int.from_bytes(raw[i * esize:(i + 1) * esize], "little", signed=signed)
        s += b
        w += (i + 1) * b
    return s & M64, w & M64


def _numpy_fp(a: np.ndarray):
    """numpy wrapping uint64 arithmetic (an independent library computation)."""
    v = a.view(VIEWS[a.itemsize]).astype(np.int64).astype(np.uint64)
    idx = np.arange(1, v.size + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return int(v.sum(dtype=np.uint64)), int((v * idx).sum(dtype=np.uint64))


@pytest.mark.parametrize("dtype", [np.uint8, np.float16, np.int16, np.float32, np.int32,
                                   np.float64, np.int64])
@pytest.mark.parametrize("n", [0, 1, 2, 7, 31, 64, 255])
def test_brute_force_tiny(dtype, n):
    rng = np.random.default_rng(n * 31 + np.dtype(dtype).itemsize)
    raw = rng.integers(0, 256, size=n * np.dtype(dtype).itemsize, dtype=np.uint8)
    a = raw.view(dtype)
    assert oracle.fingerprint(a) == _brute_fp(raw.tobytes(), a.itemsize)


@pytest.mark.parametrize("dtype", [np.uint8, np.float16, np.float32, np.float64])
def test_numpy_wrapping_sums(dtype):
    rng = np.random.default_rng(7)
    raw = rng.integers(0, 256, size=100_003 * np.dtype(dtype).itemsize, dtype=np.uint8)
    a = raw.view(dtype)
    assert oracle.fingerprint(a) == _numpy_fp(a)


def test_sign_and_zero_extension():
    # 1-byte elements are zero-extended, wider ones sign-extended
    assert oracle.fingerprint(np.array([255], dtype=np.uint8)) == (255, 255)
    assert oracle.fingerprint(np.array([-1], dtype=np.int16)) == (M64, M64)
    assert oracle.fingerprint(np.array([-2], dtype=np.int32)) == (M64 - 1, M64 - 1)
    # float32 -0.0 is 0x80000000 -> -2^31 after sign extension
    assert oracle.fingerprint(np.array([-0.0], dtype=np.float32)) == ((-(1 << 31)) & M64,) * 2


@pytest.mark.parametrize("esize,c", [(1, 0xAB), (2, -12345), (4, 0x3C23D70A), (4, -7), (8, -(1 << 62))])
@pytest.mark.parametrize("n", [1, 5, 1000, 65537])
def test_closed_form_constant(esize, c, n):
    a = np.full(n, c, dtype=VIEWS[esize])
    b = c & M64 if esize != 1 else c
    assert oracle.fingerprint(a) == ((n * b) & M64, (b * n * (n + 1) // 2) & M64)


def test_closed_form_single_nonzero():
    for i in [0, 1, 17, 999]:
        a = np.zeros(1000, dtype=np.int32)
        a[i] = -123456
        assert oracle.fingerprint(a) == ((-123456) & M64, (-123456 * (i + 1)) & M64)
    assert oracle.fingerprint(np.zeros(4096, dtype=np.float32)) == (0, 0)


def test_slices_match_single_walk():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(3_000_001).astype(np.float32)
    assert oracle.fingerprint(a, threads=4) == oracle.fingerprint(a, threads=1)


def test_concatenation_identity():
    # fingerprint(a || b) = (S_a + S_b, W_a + W_b + len(a) * S_b): positions continue
    rng = np.random.default_rng(4)
    a = rng.standard_normal(1000).astype(np.float32)
    b = rng.standard_normal(333).astype(np.float32)
    sa, wa = oracle.fingerprint(a)
    sb, wb = oracle.fingerprint(b)
    assert oracle.fingerprint(np.concatenate([a, b])) == ((sa + sb) & M64, (wa + wb + len(a) * sb) & M64)


@pytest.mark.parametrize("dtype", [np.uint8, np.float16, np.float32, np.float64])
def test_every_single_bit_flip_changes_plain_sum(dtype):
    # flipping bit k changes the widened value by +-2^k (or +-2^k with sign extension): != 0 mod 2^64
    rng = np.random.default_rng(5)
    a = rng.integers(0, 256, size=64 * np.dtype(dtype).itemsize, dtype=np.uint8).view(dtype).copy()
    s0, _ = oracle.fingerprint(a)
    u = a.view(np.uint8)
    for elem in [0, 13, 63]:
        for bit in range(8 * a.itemsize):
            b = u.copy()
            b[elem * a.itemsize + bit // 8] ^= 1 << (bit % 8)
            assert oracle.fingerprint(b.view(dtype))[0] != s0


def test_two_element_guarantee_exhaustive_small():
    # the page's guarantee: any change to 1 or 2 elements changes (S, W) when numel < 2^32, esize <= 4
    rng = np.random.default_rng(6)
    n = 24
    base = rng.integers(-(1 << 31), 1 << 31, size=n, dtype=np.int64).astype(np.int32)
    fp0 = oracle.fingerprint(base)
    for i in range(n):
        for j in range(i, n):
            for _ in range(3):
                b = base.copy()
                d = int(rng.integers(1, 1 << 20))
                b[i] = np.int32((int(b[i]) + d + (1 << 31)) % (1 << 32) - (1 << 31))
                if j != i:  # compensating change: plain sum unchanged on purpose
                    b[j] = np.int32((int(b[j]) - d + (1 << 31)) % (1 << 32) - (1 << 31))
                if np.array_equal(b, base):
                    continue
                assert oracle.fingerprint(b) != fp0


def test_two_element_guarantee_random_large():
    rng = np.random.default_rng(8)
    n = 5_000_000
    base = rng.integers(-(1 << 15), 1 << 15, size=n, dtype=np.int64).astype(np.int16)
    fp0 = oracle.fingerprint(base)
    for _ in range(20):
        i, j = sorted(rng.choice(n, size=2, replace=False).tolist())
        b = base.copy()
        b[i], b[j] = base[j], base[i]
        if b[i] == base[i]:
            continue
        s, w = oracle.fingerprint(b)
        assert s == fp0[0] and w != fp0[1]


def test_pages_weight_faults():
    g = json.load(open(os.path.join(GOLDEN, "weight_faults.json")))
    rng = np.random.default_rng(9)
    w = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    s0, w0 = oracle.fingerprint(w)
    for f in g["faults"]:
        x = w.copy()
        u = x.view(np.uint32)
        if f["kind"] == "bit_flip":
            u[100] ^= np.uint32(1 << f["bit"])
        elif f["kind"] == "swap":
            x[10], x[20] = w[20], w[10]
        else:
            u[10] = np.uint32((int(u[10]) + f["deltas"][0]) % (1 << 32))
            u[20] = np.uint32((int(u[20]) + f["deltas"][1]) % (1 << 32))
        s1, w1 = oracle.fingerprint(x)
        assert (s1 != s0) == f["plain_sum_changes"], f["kind"]
        assert (w1 != w0) == f["weighted_sum_changes"], f["kind"]


# ---------------------------------------------------------------- xorsum
@pytest.mark.parametrize("dtype", [np.uint8, np.float16, np.float32, np.float64])
def test_xorsum_brute_force(dtype):
    rng = np.random.default_rng(10)
    raw = rng.integers(0, 256, size=333 * np.dtype(dtype).itemsize, dtype=np.uint8)
    a = raw.view(dtype)
    es = a.itemsize
    ref = reduce(lambda x, y: x ^ y,
                 (int.from_bytes(raw[i * es:(i + 1) * es].tobytes(), "little") for i in range(a.size)), 0)
    assert oracle.xorsum(a) == ref
    unsigned = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[es]
    assert oracle.xorsum(a) == int(np.bitwise_xor.reduce(a.view(unsigned)))


def test_xorsum_linearity_and_collisions():
    rng = np.random.default_rng(11)
    a = rng.integers(0, 1 << 16, size=1001, dtype=np.uint16)
    b = rng.integers(0, 1 << 16, size=1001, dtype=np.uint16)
    assert oracle.xorsum(a) ^ oracle.xorsum(b) == oracle.xorsum(a ^ b)
    assert oracle.xorsum(np.zeros(0, dtype=np.uint16)) == 0
    # a single bit flip shows up exactly at its bit position
    c = a.copy()
    c[500] ^= 1 << 9
    assert oracle.xorsum(a) ^ oracle.xorsum(c) == 1 << 9
    # the same bit flipped in two elements cancels: the collision the review page notes
    c[700] ^= 1 << 9
    assert oracle.xorsum(c) == oracle.xorsum(a)
    assert oracle.xorsum_compare([1, 2, 3], [1, 6, 3]) == ([0, 1, 0], [0, 4, 0])
