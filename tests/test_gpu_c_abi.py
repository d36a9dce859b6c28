"""The C ABI from C: two plain C programs include include/sdc.h and link
libsdc.so and the CUDA runtime, with no Python or torch on their path.
tests/c_abi_fingerprint.c fingerprints and votes on replicas this test writes
to a file; what it prints must equal the oracle on the same bytes.
tests/c_abi_abft.c runs the GEMM checksum path (product with row and column
checksums, verifier, the fused row check, capture and pair replay) on operands
this test writes; what it prints is compared with the oracle.

Sources: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" (AWS Machine Learning Blog), "Compare by fingerprint" and
"Check 3: Weight fingerprints, after the optimizer step"; "Safeguarding LLM
Training at Scale: Online SDC Detection and Insights from 35 Million GPU Hours"
(review page), method sections 1 and 2.
"""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def c_program(tmp_path_factory):
    import silent_corruption_checksums_gb300 as sdc  # builds the library if it is stale
    lib_dir = os.path.dirname(sdc.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_fingerprint")
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "no C compiler"
    subprocess.run([cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA_HOME, "include"), os.path.join(HERE, "c_abi_fingerprint.c"), "-o", exe,
                    "-L", lib_dir, "-lsdc", "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA_HOME, 'lib64')}"], check=True)
    return exe


def _replicas(seed):
    """3 replicas of 6 tensors of every element width (an empty one, odd lengths); replica 1
    has one bit flipped in tensor 2, replica 2 one element changed in tensor 4."""
    rng = np.random.default_rng(seed)
    shapes = [(1, 1000), (2, 777), (4, 4099), (8, 33), (4, 0), (2, 65536 + 3)]
    base = [rng.integers(0, 256, n * esize, dtype=np.uint8) for esize, n in shapes]
    reps = [[b.copy() for b in base] for _ in range(3)]
    reps[1][2][5] ^= 0x10
    reps[2][5][7] ^= 0xFF
    return shapes, reps


def _views(shapes, rep):
    kinds = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}
    return [b.view(kinds[esize]) for (esize, _), b in zip(shapes, rep)]


def test_c_caller_matches_the_oracle(c_program, tmp_path):
    shapes, reps = _replicas(21)
    path = tmp_path / "input.bin"
    with open(path, "wb") as f:
        f.write(struct.pack("<II", len(reps), len(shapes)))
        for esize, n in shapes:
            f.write(struct.pack("<QI", n, esize))
        for rep in reps:
            for b in rep:
                f.write(b.tobytes())
    out = subprocess.run([c_program, str(path)], check=True, capture_output=True, text=True).stdout.split("\n")
    fp = {}
    suspects = {}
    summary = None
    for line in out:
        f = line.split()
        if not f:
            continue
        if f[0] == "fp":
            fp[(int(f[1]), int(f[2]))] = (int(f[3], 16), int(f[4], 16))
        elif f[0] == "suspect":
            suspects[int(f[1])] = (int(f[2]), int(f[3], 16))
        elif f[0] == "summary":
            summary = {"diverged": int(f[1]), "no_majority": int(f[2]), "suspect_mask": int(f[3], 16)}
    table = [[oracle.fingerprint(v) for v in _views(shapes, rep)] for rep in reps]
    for r in range(len(reps)):
        for t in range(len(shapes)):
            assert fp[(r, t)] == table[r][t], (r, t)
    suspect, mask, summ = oracle.vote(table)
    for t in range(len(shapes)):
        assert suspects[t] == (suspect[t], mask[t]), t
    assert summary == summ
    assert summ == {"diverged": 1, "no_majority": 0, "suspect_mask": 0b110}


@pytest.fixture(scope="module")
def c_abft_program(tmp_path_factory):
    import silent_corruption_checksums_gb300 as sdc
    lib_dir = os.path.dirname(sdc.LIB_PATH)
    exe = str(tmp_path_factory.mktemp("c_abi") / "c_abi_abft")
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "no C compiler"
    subprocess.run([cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(CUDA_HOME, "include"), os.path.join(HERE, "c_abi_abft.c"), "-o", exe,
                    "-L", lib_dir, "-lsdc", "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA_HOME, 'lib64')}"], check=True)
    return exe


def _bf16_bits(rng, shape, std):
    """Seeded bfloat16 bits of N(0, std^2) values (rounded to nearest even from float32)."""
    x = (rng.standard_normal(shape) * std).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((x + 0x7FFF + ((x >> 16) & 1)) >> 16).astype(np.uint16)


def _run_abft(exe, tmp_path, A, Wb, Wp):
    M, K = A.shape
    N = Wb.shape[0]
    path, cpath = tmp_path / "abft.bin", tmp_path / "c.bin"
    with open(path, "wb") as f:
        f.write(struct.pack("<III", M, N, K))
        for a in (A, Wb, Wp):
            f.write(np.ascontiguousarray(a).tobytes())
    out = subprocess.run([exe, str(path), str(cpath)], check=True, capture_output=True, text=True).stdout
    r = {"rowsum": np.zeros(M), "colsum": np.zeros(N), "flag": set(), "flagcol": set(), "checkedflag": set(),
         "rowidx": {}, "colidx": {}, "differs": np.zeros((4, 4), np.uint8)}
    for line in out.split("\n"):
        f = line.split()
        if not f:
            continue
        if f[0] in ("rowsum", "colsum"):
            r[f[0]][int(f[1])] = float.fromhex(f[2])
        elif f[0] in ("flag", "flagcol", "checkedflag"):
            r[f[0]].add(int(f[1]))
        elif f[0] in ("rowidx", "colidx"):
            r[f[0]][int(f[1])] = int(f[2])
        elif f[0] == "differs":
            r["differs"][int(f[1]), int(f[2])] = int(f[3])
        else:
            r[f[0]] = [int(v) for v in f[1:]]
    r["C"] = np.fromfile(cpath, dtype=np.uint16).reshape(M, N)
    return r


@pytest.mark.parametrize("fault", [False, True])
def test_c_caller_gemm_checksum_path(c_abft_program, tmp_path, fault):
    # C = A W^T through the C ABI alone: the checksums within the oracle's rounding bound of the
    # exact sums, the verifier's and the fused check's flags where the oracle's residual clearly
    # decides, the capture of the verifier's flags equal to the oracle's, the pair replay equal to
    # the oracle's consistency verdict.  The fault: one weight of W's rows 100 and 700 has its top
    # exponent bit flipped for the product while the check trusts the clean W.
    M, N, K = 300, 776, 520
    rng = np.random.default_rng(61)
    A, Wb = _bf16_bits(rng, (M, K), 1.0), _bf16_bits(rng, (N, K), 0.02)
    Wp = Wb.copy()
    if fault:
        for j in (100, 700):
            Wp[j, int(rng.integers(0, K))] ^= 0x4000
    r = _run_abft(c_abft_program, tmp_path, A, Wb, Wp)
    assert r["gemm"] == [0] and r["checked"][0] == 0 and r["checked"][3] == 1  # no abort; the same C bits
    exact = oracle.abft_product(A, Wp)
    _, mag = oracle.abft_reference(A, Wp)
    _, mag_col = oracle.abft_reference_cols(A, Wp)
    assert np.all(np.abs(r["rowsum"] - exact.sum(axis=1)) <= oracle.abft_bound(mag, N, K))
    assert np.all(np.abs(r["colsum"] - exact.sum(axis=0)) <= oracle.abft_bound(mag_col, M, K))
    v = oracle.abft_verify(exact.sum(axis=1), A, Wb)
    vc = oracle.abft_verify_cols(exact.sum(axis=0), A, Wb)
    for res, bnd, got in ((v["residual"], v["bound"], r["flag"]), (v["residual"], v["bound"], r["checkedflag"]),
                          (vc["residual"], vc["bound"], r["flagcol"])):
        clear = set(np.nonzero(np.abs(res) > 2.0 * bnd)[0].tolist())
        clean = set(np.nonzero(np.abs(res) <= 1e-6 * bnd)[0].tolist())
        assert clear <= got and not (clean & got)
    assert r["verify"] == [len(r["flag"]), len(r["flagcol"])] and r["checked"][1:3] == [len(r["checkedflag"]), 0]
    flag = np.isin(np.arange(M), sorted(r["flag"])).astype(np.uint8)
    flag_col = np.isin(np.arange(N), sorted(r["flagcol"])).astype(np.uint8)
    ref = oracle.abft_capture(flag, flag_col, A, Wb, r["C"], 4, 4)
    assert r["capture"] == [ref["n_rows"], ref["n_cols"]]
    assert [r["rowidx"][i] for i in range(len(ref["row_idx"]))] == ref["row_idx"].tolist()
    assert [r["colidx"][i] for i in range(len(ref["col_idx"]))] == ref["col_idx"].tolist()
    want = np.zeros((4, 4), np.uint8)
    if len(ref["row_idx"]) and len(ref["col_idx"]):
        want[:len(ref["row_idx"]), :len(ref["col_idx"])] = oracle.abft_replay_pairs(ref)
    assert np.array_equal(r["differs"], want) and r["replay"] == [int(want.sum()), 0]
    if fault:
        assert r["flagcol"] == {100, 700} and len(r["flag"]) >= M // 2 and want.sum() == 8
    else:
        assert not r["flag"] and not r["flagcol"] and not r["checkedflag"] and r["capture"] == [0, 0]
