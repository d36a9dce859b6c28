"""The bounded barrier wait gives up on a phase nothing completes and reports it,
then succeeds once the phase completes: the failure path of the TMA and
tensor-core kernels, made to run out on purpose without faulting or hanging."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


@pytest.mark.parametrize("polls", [1, 1000, 100_000])
def test_bounded_wait_gives_up_then_succeeds(sdc, polls):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    sdc.sdc_selftest_bounded_wait(polls, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status[0]) == 3
    assert time.perf_counter() - t0 < 30.0
    # the context is still usable
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


def test_rejects_bad_arguments(sdc):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for polls, code in [(0, 9), (1 << 25, 9)]:
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_selftest_bounded_wait(polls, status.data_ptr(), 0)
        assert ei.value.status == code
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_selftest_bounded_wait(10, 0, 0)
    assert ei.value.status == 1
