"""The C ABI from C: tests/c_abi_fingerprint.c includes include/sdc.h, links
libsdc.so and the CUDA runtime, and fingerprints and votes on replicas this test
writes to a file; what it prints must equal the oracle on the same bytes.

Sources: "Detecting and recovering from silent data corruption on Amazon
SageMaker HyperPod" (AWS Machine Learning Blog), "Compare by fingerprint" and
"Check 3: Weight fingerprints, after the optimizer step".
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
