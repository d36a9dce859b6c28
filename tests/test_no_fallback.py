"""There is no CPU fallback: without the compiled library every call raises,
and the binding refuses host tensors instead of fingerprinting them on the
CPU.  (Each case runs in a child interpreter, so the module state of the other
tests is untouched.)"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code: str) -> subprocess.CompletedProcess:
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)


def test_missing_library_makes_every_call_raise():
    r = _run("""
import silent_corruption_checksums_gb300 as s
s.LIB_PATH = 'no-such-dir/libsdc.so'
s._lib = s._Missing(ImportError('missing'))
for call in (lambda: s.sdc_status_string(0), lambda: s.sdc_workspace_size(None),
             lambda: s.sdc_abft_workspace_size(128, 256, 64)):
    try:
        call()
    except ImportError as e:
        assert 'libsdc.so not found' in str(e), e
    else:
        raise SystemExit('a call returned without the library')
print('ok')
""")
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_host_tensors_are_refused():
    pytest.importorskip("torch")
    r = _run("""
import torch
import silent_corruption_checksums_gb300 as s
try:
    s.Plan([[torch.zeros(16)], [torch.zeros(16)]])
except ValueError as e:
    assert 'CUDA tensors' in str(e), e
    print('ok')
else:
    raise SystemExit('a plan over host tensors was accepted')
""")
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
