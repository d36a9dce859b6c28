"""Seeded synthetic inputs for the replica-integrity scan.

Shared by the tests and the benchmark; used by both the CUDA path and the
oracle (which receives host copies).  This module holds none of the method's
arithmetic: it only lays out tensors, draws seeded values and injects faults,
recording each injection as ground truth.

Workloads (sizes follow the parameter layouts below):
  tiny      3 replicas of 4 float32 tensors (64x32, 32, 128x64, 10), N(0, 0.02);
            replica 1 gets one seeded bit flip.
  1b        ~1.04e9-parameter transformer layout (24 layers, d=1792,
            ffn=7168, vocab=32000, untied embedding and head), float32
            N(0, 0.02), 3 replicas, one seeded bit flip in one replica.
  grad      the 1b layout as 4 flat bf16 local-gradient buffers N(0, 1e-3),
            each seeded separately; buffer 2 gets NaN / +Inf / -Inf / +-2^70
            at rate 1e-7.
  8b        Llama-style layout (32 layers, d=4096, 8 kv heads of 128,
            ffn=14336, vocab=128256), bf16 N(0, 0.02), 8 replicas; one
            replica gets 16 elements XORed with non-zero 16-bit masks.
  gemm      a linear layer's forward product C = A W^T: A [M, K] bf16 N(0, 1)
            activations, W [N, K] bf16 N(0, 0.02) weights; the benchmark
            shape is the 8b layout's MLP up-projection (M = 8192 tokens,
            N = 14336, K = 4096).  A fault is planted by XORing bits of chosen
            elements of a copy of A (the operand as a faulty unit would read
            it), the clean A being the reference.
  attn      one attention layer's backward inputs: BH heads of L tokens, head
            dimension 128, Q, K, dO bf16 N(0, 1), scale 1/sqrt(128), and the
            forward's log-sum-exp (torch.logsumexp of the float32 scores, the
            causal mask applied) as float32; the benchmark shape is the 8b
            layout's 32 heads at L = 4096, causal.  Faults are planted in a
            copy of an input (a shifted log-sum-exp row, an XORed element of K).
  stress    100,000 tensors, numel = floor(exp(U(0, ln(1e6 + 1)))), dtype
            uniform over float32/bf16/float16, packed per replica in one flat
            buffer (element-aligned starts), 3 replicas with one bit flip;
            plus 1,000 (original, recomputed) pairs for the xorsum compare,
            a seeded half of which differ in one bit.
"""
from __future__ import annotations

import math

import numpy as np
import torch

# ---------------------------------------------------------------- layouts
def layout_1b(layers: int = 24) -> list[tuple[str, tuple[int, ...]]]:
    d, ffn, vocab = 1792, 7168, 32000
    out = [("embed", (vocab, d))]
    for i in range(layers):
        out += [(f"l{i}.q", (d, d)), (f"l{i}.k", (d, d)), (f"l{i}.v", (d, d)), (f"l{i}.o", (d, d)),
                (f"l{i}.up", (ffn, d)), (f"l{i}.down", (d, ffn)), (f"l{i}.norm1", (d,)), (f"l{i}.norm2", (d,))]
    out += [("final_norm", (d,)), ("head", (vocab, d))]
    return out


def layout_8b(layers: int = 32) -> list[tuple[str, tuple[int, ...]]]:
    d, kv, ffn, vocab = 4096, 1024, 14336, 128256
    out = [("embed", (vocab, d))]
    for i in range(layers):
        out += [(f"l{i}.q", (d, d)), (f"l{i}.k", (kv, d)), (f"l{i}.v", (kv, d)), (f"l{i}.o", (d, d)),
                (f"l{i}.gate", (ffn, d)), (f"l{i}.up", (ffn, d)), (f"l{i}.down", (d, ffn)),
                (f"l{i}.norm1", (d,)), (f"l{i}.norm2", (d,))]
    out += [("final_norm", (d,)), ("head", (vocab, d))]
    return out


TINY_SHAPES = [(64, 32), (32,), (128, 64), (10,)]


def numel_of(shape) -> int:
    return int(math.prod(shape))


def layout_numel(layout) -> int:
    return sum(numel_of(s) for _, s in layout)


# ---------------------------------------------------------------- primitives
_INT_VIEW = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}


def normal(shape, std: float, dtype, gen: torch.Generator, device) -> torch.Tensor:
    """N(0, std) drawn in float32 and rounded to dtype."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


def xor_element(t: torch.Tensor, flat_index: int, mask: int) -> None:
    """XOR the raw bits of one element (flat row-major index) with `mask`, in place."""
    es = t.element_size()
    bits = t.view(-1).view(_INT_VIEW[es])
    width = 8 * es
    m = mask & ((1 << width) - 1)
    if es > 1 and m >= 1 << (width - 1):
        m -= 1 << width  # two's complement value of the mask in the signed view
    bits[flat_index : flat_index + 1].bitwise_xor_(m)


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


# ---------------------------------------------------------------- workloads
def replicas_from(base: list[torch.Tensor], n: int) -> list[list[torch.Tensor]]:
    return [[t.clone() for t in base] for _ in range(n)]


def tiny(device="cpu", seed: int = 0) -> dict:
    g = generator(seed, device)
    base = [normal(s, 0.02, torch.float32, g, device) for s in TINY_SHAPES]
    reps = replicas_from(base, 3)
    rng = np.random.default_rng(seed)
    k = int(rng.integers(len(TINY_SHAPES)))
    e = int(rng.integers(numel_of(TINY_SHAPES[k])))
    bit = int(rng.integers(32))
    xor_element(reps[1][k], e, 1 << bit)
    return {"replicas": reps, "truth": {"replica": 1, "tensor": k, "element": e, "bit": bit}}


def worked_example(device="cpu", fault: bool = False) -> dict:
    """The page's three-replica SGD example as float32 scalars: (weights, local gradients, lr)."""
    grads = [0.20, 4.00 if fault else 0.40, 0.30]
    return {"weights": [torch.tensor([0.500], dtype=torch.float32, device=device) for _ in range(3)],
            "grads": [torch.tensor([v], dtype=torch.float32, device=device) for v in grads],
            "lr": 0.1}


def weights(layout, n_replicas: int, dtype, std: float, device, seed: int) -> list[list[torch.Tensor]]:
    g = generator(seed, device)
    base = [normal(s, std, dtype, g, device) for _, s in layout]
    reps = [base] + [[t.clone() for t in base] for _ in range(n_replicas - 1)]
    return reps


def weights_1b(device, seed: int = 1, n_replicas: int = 3, n_layers: int = 24) -> dict:
    layout = layout_1b(n_layers)
    reps = weights(layout, n_replicas, torch.float32, 0.02, device, seed)
    rng = np.random.default_rng(seed)
    r = int(rng.integers(n_replicas))
    k = int(rng.integers(len(layout)))
    e = int(rng.integers(numel_of(layout[k][1])))
    bit = int(rng.integers(32))
    xor_element(reps[r][k], e, 1 << bit)
    return {"replicas": reps, "layout": layout,
            "truth": {"replica": r, "tensor": k, "element": e, "bit": bit}}


GRAD_KINDS = ("nan", "+inf", "-inf", "+2^70", "-2^70")
_GRAD_KIND_VALUES = {"nan": float("nan"), "+inf": float("inf"), "-inf": float("-inf"),
                     "+2^70": 2.0 ** 70, "-2^70": -(2.0 ** 70)}


def grads_flat(numel: int, n_bufs: int, dtype, std: float, device, seed: int, inject_buf: int = 2,
               rate: float = 1e-7, min_injections: int = 0) -> dict:
    """n_bufs flat local-gradient buffers; buffer `inject_buf` gets seeded non-finite/huge values."""
    bufs = [normal((numel,), std, dtype, generator(seed + 1000 * b, device), device) for b in range(n_bufs)]
    rng = np.random.default_rng(seed)
    n_inj = max(min_injections, int(rng.binomial(numel, rate))) if numel else 0
    n_inj = min(n_inj, numel)
    pos = np.sort(rng.choice(numel, size=n_inj, replace=False)) if n_inj else np.zeros(0, dtype=np.int64)
    kinds = rng.integers(0, len(GRAD_KINDS), size=n_inj)
    truth = []
    if n_inj and 0 <= inject_buf < n_bufs:
        vals = torch.tensor([_GRAD_KIND_VALUES[GRAD_KINDS[k]] for k in kinds], dtype=torch.float32,
                            device=device).to(dtype)
        bufs[inject_buf][torch.as_tensor(pos, device=device)] = vals
        truth = [(int(p), GRAD_KINDS[int(k)]) for p, k in zip(pos, kinds)]
    return {"bufs": bufs, "truth": truth, "inject_buf": inject_buf}


def grads_1b(device, seed: int = 3) -> dict:
    return grads_flat(layout_numel(layout_1b()), 4, torch.bfloat16, 1e-3, device, seed)


def weights_8b(device, seed: int = 4, n_replicas: int = 8, n_layers: int = 32) -> dict:
    layout = layout_8b(n_layers)
    reps = weights(layout, n_replicas, torch.bfloat16, 0.02, device, seed)
    rng = np.random.default_rng(seed)
    r = int(rng.integers(n_replicas))
    k = int(rng.integers(len(layout)))
    n = numel_of(layout[k][1])
    elems = np.sort(rng.choice(n, size=min(16, n), replace=False))
    masks = rng.integers(1, 1 << 16, size=len(elems))
    for e, m in zip(elems, masks):
        xor_element(reps[r][k], int(e), int(m))
    return {"replicas": reps, "layout": layout,
            "truth": {"replica": r, "tensor": k, "elements": elems.tolist(), "masks": masks.tolist()}}


_STRESS_DTYPES = (torch.float32, torch.bfloat16, torch.float16)


def stress_sizes(n_tensors: int, seed: int, max_numel: int = 1_000_000):
    rng = np.random.default_rng(seed)
    numel = np.floor(np.exp(rng.uniform(0.0, math.log(max_numel + 1), size=n_tensors))).astype(np.int64)
    numel = np.clip(numel, 1, max_numel)
    dt = rng.integers(0, 3, size=n_tensors)
    return numel, dt


def _packed(numel, dt, device, gen, std=0.02):
    """One flat byte buffer holding the tensors back to back (element-aligned), and views into it."""
    sizes = [int(n) * _STRESS_DTYPES[int(d)].itemsize for n, d in zip(numel, dt)]
    offs = []
    o = 0
    for s, d in zip(sizes, dt):
        es = _STRESS_DTYPES[int(d)].itemsize
        o = (o + es - 1) // es * es
        offs.append(o)
        o += s
    flat = torch.empty(max(o, 16), dtype=torch.uint8, device=device)
    # values: one float32 draw per dtype group, rounded and copied into place
    for di, dtype in enumerate(_STRESS_DTYPES):
        idx = [i for i in range(len(numel)) if int(dt[i]) == di]
        total = sum(int(numel[i]) for i in idx)
        if not total:
            continue
        vals = normal((total,), std, dtype, gen, device)
        s = 0
        for i in idx:
            n = int(numel[i])
            flat[offs[i] : offs[i] + n * dtype.itemsize].view(dtype).copy_(vals[s : s + n])
            s += n
        del vals
    views = [flat[offs[i] : offs[i] + int(numel[i]) * _STRESS_DTYPES[int(dt[i])].itemsize].view(
        _STRESS_DTYPES[int(dt[i])]) for i in range(len(numel))]
    return flat, views, offs


def stress(device, seed: int = 5, n_tensors: int = 100_000, n_replicas: int = 3, n_pairs: int = 1000,
           max_numel: int = 1_000_000) -> dict:
    numel, dt = stress_sizes(n_tensors, seed, max_numel)
    flat0, views0, offs = _packed(numel, dt, device, generator(seed, device))
    flats = [flat0] + [flat0.clone() for _ in range(n_replicas - 1)]
    reps = []
    for f in flats:
        reps.append([f[offs[i] : offs[i] + int(numel[i]) * _STRESS_DTYPES[int(dt[i])].itemsize].view(
            _STRESS_DTYPES[int(dt[i])]) for i in range(n_tensors)])
    rng = np.random.default_rng(seed + 1)
    r = int(rng.integers(n_replicas))
    k = int(rng.integers(n_tensors))
    e = int(rng.integers(int(numel[k])))
    bit = int(rng.integers(8 * _STRESS_DTYPES[int(dt[k])].itemsize))
    xor_element(reps[r][k], e, 1 << bit)
    # xorsum pairs: originals and their "recomputed" copies
    pnumel, pdt = stress_sizes(n_pairs, seed + 2, max_numel)
    pflat, orig, poffs = _packed(pnumel, pdt, device, generator(seed + 2, device))
    rflat = pflat.clone()
    recomp = [rflat[poffs[i] : poffs[i] + int(pnumel[i]) * _STRESS_DTYPES[int(pdt[i])].itemsize].view(
        _STRESS_DTYPES[int(pdt[i])]) for i in range(n_pairs)]
    differ = np.sort(rng.choice(n_pairs, size=n_pairs // 2, replace=False))
    pair_truth = []
    for p in differ:
        es = _STRESS_DTYPES[int(pdt[p])].itemsize
        ee = int(rng.integers(int(pnumel[p])))
        bb = int(rng.integers(8 * es))
        xor_element(recomp[p], ee, 1 << bb)
        pair_truth.append((int(p), ee, bb))
    return {"replicas": reps, "flats": flats, "numel": numel, "dtypes": dt,
            "truth": {"replica": r, "tensor": k, "element": e, "bit": bit},
            "pairs": {"orig": orig, "recomp": recomp, "flats": (pflat, rflat), "differ": pair_truth}}


GEMM_8B_UP = (8192, 14336, 4096)  # tokens, ffn, d of the 8b layout


def gemm_operands(M: int, N: int, K: int, device, seed: int = 6, a_std: float = 1.0, w_std: float = 0.02) -> dict:
    """Seeded bf16 A [M, K] (activations) and W [N, K] (weights)."""
    gen = generator(seed, device)
    A = normal((M, K), a_std, torch.bfloat16, gen, device)
    W = normal((N, K), w_std, torch.bfloat16, gen, device)
    return {"A": A, "W": W}


def wgrad_operands(T: int, N: int, K: int, device, seed: int = 10, dy_std: float = 2.0 ** -10,
                   x_std: float = 1.0) -> dict:
    """Seeded bf16 dY [T, N] (a linear layer's output gradient) and X [T, K] (its input),
    token-major: the operands of its weight gradient dW = dY^T X."""
    gen = generator(seed, device)
    dY = normal((T, N), dy_std, torch.bfloat16, gen, device)
    X = normal((T, K), x_std, torch.bfloat16, gen, device)
    return {"dY": dY, "X": X}


def gemm_fault(A: torch.Tensor, rows: list[int], seed: int = 7, mask: int = 0x4000) -> tuple[torch.Tensor, list]:
    """A copy of A with one seeded element of each listed row XORed with `mask`
    (default: the top exponent bit of a bf16).  Returns (faulty A, [(row, col)])."""
    rng = np.random.default_rng(seed)
    Af = A.clone()
    K = A.shape[1]
    where = []
    for r in rows:
        c = int(rng.integers(0, K))
        xor_element(Af, r * K + c, mask)
        where.append((int(r), c))
    return Af, where


ATTN_8B = (32, 4096)  # heads, tokens (head dimension 128)


def attn_inputs(BH: int, L: int, device, seed: int = 8, causal: bool = True, D: int = 128, group: int = 1) -> dict:
    """Seeded Q, dO (bf16 [BH, L, D]), K (bf16 [BH / group, L, D]: query head h uses
    K/V head h / group) and the forward's float32 log-sum-exp [BH, L]."""
    gen = generator(seed, device)
    Q = normal((BH, L, D), 1.0, torch.bfloat16, gen, device)
    K = normal((BH // group, L, D), 1.0, torch.bfloat16, gen, device)
    dO = normal((BH, L, D), 1.0, torch.bfloat16, gen, device)
    scale = 1.0 / math.sqrt(D)
    lse = torch.empty((BH, L), dtype=torch.float32, device=device)
    # the forward's softmax statistics, one head at a time; past 8,192 tokens, in blocks of
    # 4,096 query rows (the whole score matrix of a head would not fit)
    rows = L if L <= 8192 else 4096
    for h in range(BH):
        Kf = K[h // group].float()
        for r0 in range(0, L, rows):
            s = (Q[h, r0:r0 + rows].float() @ Kf.t()) * scale
            if causal:
                keys = torch.arange(L, device=device)[None, :]
                qs = torch.arange(r0, min(L, r0 + rows), device=device)[:, None]
                s.masked_fill_(keys > qs, float("-inf"))
            lse[h, r0:r0 + rows] = torch.logsumexp(s, dim=-1)
    return {"Q": Q, "K": K, "dO": dO, "lse": lse, "scale": scale, "causal": causal, "group": group}
