"""The allocation-free average-scan entry point, called through the C ABI,
agrees with the regular entry point (which takes a caller-allocated
workspace) on two calls in a row, and rejects sizes beyond its fixed scratch.

This file is collected last on purpose: the entry point shares one
library-wide scratch array, and the test must pass both alone in a fresh
process and after every other test has run.
"""
import numpy as np
import pytest
import torch

import sdc_workloads as W
from tests._helpers import host_bits, stats_match

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sdc():
    import silent_corruption_checksums_gb300 as m
    return m


def _stats_tensors(n_bufs):
    pre = torch.empty((n_bufs, 56), dtype=torch.uint8, device=DEV)
    post = torch.empty(56, dtype=torch.uint8, device=DEV)
    return pre, post


@pytest.mark.parametrize("dtype,code", [(torch.bfloat16, 2), (torch.float32, 1), (torch.float16, 3)])
def test_matches_workspace_entry_point_twice(sdc, dtype, code):
    numel = 3 * 8192 * 7 + 13
    g = W.grads_flat(numel, 4, dtype, 1e-3, DEV, seed=31, rate=1e-3)
    bufs = g["bufs"]
    ptrs = [b.data_ptr() for b in bufs]
    stream = torch.cuda.current_stream().cuda_stream
    # regular entry point, caller-provided workspace
    need = sdc.sdc_grad_average_scan_workspace_size(numel, 4, code)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    ref_avg = torch.empty_like(bufs[0])
    ref_pre, ref_post = _stats_tensors(4)
    sdc.sdc_grad_average_scan(ptrs, ref_avg.data_ptr(), numel, code, ref_pre.data_ptr(), ref_post.data_ptr(),
                              ws.data_ptr(), need, stream)
    torch.cuda.synchronize()
    ref_pre_d, ref_post_d = sdc.decode_stats(ref_pre), sdc.decode_stats(ref_post)[0]
    for _ in range(2):  # two calls in a row share the static scratch
        avg = torch.full_like(bufs[0], 7.0)
        pre, post = _stats_tensors(4)
        pre.fill_(0xAB)
        post.fill_(0xAB)
        sdc.sdc_grad_average_scan_noalloc(ptrs, avg.data_ptr(), numel, code, pre.data_ptr(), post.data_ptr(),
                                          stream)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(avg), host_bits(ref_avg))
        for b, st in enumerate(sdc.decode_stats(pre)):
            stats_match(st, ref_pre_d[b])
        stats_match(sdc.decode_stats(post)[0], ref_post_d)


def test_rejects_sizes_beyond_the_scratch(sdc):
    small = [torch.zeros(16, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    out = torch.empty_like(small[0])
    pre, post = _stats_tensors(4)
    too_many = 2 ** 31  # elements: far more partials than 16 MiB holds
    assert sdc.sdc_grad_average_scan_workspace_size(too_many, 4, 2) > sdc.NOALLOC_SCRATCH_BYTES
    with pytest.raises(sdc.SdcError) as ei:
        sdc.sdc_grad_average_scan_noalloc([b.data_ptr() for b in small], out.data_ptr(), too_many, 2,
                                          pre.data_ptr(), post.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == 9
    assert "static scratch" in sdc.sdc_last_error()


def _call_both(sdc, bufs, code):
    """The regular entry point (own workspace) and the allocation-free one on the same inputs."""
    n_bufs, numel = len(bufs), bufs[0].numel()
    ptrs = [b.data_ptr() for b in bufs]
    stream = torch.cuda.current_stream().cuda_stream
    need = sdc.sdc_grad_average_scan_workspace_size(numel, n_bufs, code)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=DEV)
    ref_avg, got_avg = torch.empty_like(bufs[0]), torch.full_like(bufs[0], 7.0)
    ref_pre, ref_post = _stats_tensors(n_bufs)
    pre, post = _stats_tensors(n_bufs)
    pre.fill_(0xAB)
    post.fill_(0xAB)
    sdc.sdc_grad_average_scan(ptrs, ref_avg.data_ptr(), numel, code, ref_pre.data_ptr(), ref_post.data_ptr(),
                              ws.data_ptr(), need, stream)
    sdc.sdc_grad_average_scan_noalloc(ptrs, got_avg.data_ptr(), numel, code, pre.data_ptr(), post.data_ptr(), stream)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(got_avg), host_bits(ref_avg))
    for got, ref in zip(sdc.decode_stats(pre), sdc.decode_stats(ref_pre)):
        stats_match(got, ref, rtol=0.0)
    stats_match(sdc.decode_stats(post)[0], sdc.decode_stats(ref_post)[0], rtol=0.0)


def test_smaller_call_after_a_larger_one(sdc):
    # the scratch keeps the last call's partials and group sums: a large, NaN-heavy call with
    # 8 buffers leaves non-zero counts in it, and a later, smaller call with 2 buffers must
    # not see any of them (every partial it reads is written by that call first)
    big = W.grads_flat(40 * 8192 + 3, 8, torch.bfloat16, 1e-3, DEV, seed=33, rate=2e-2)["bufs"]
    _call_both(sdc, big, 2)
    small = W.grads_flat(5 * 8192 + 1, 2, torch.bfloat16, 1e-3, DEV, seed=34)["bufs"]
    _call_both(sdc, small, 2)
    _call_both(sdc, big[:3], 2)


def test_size_limit_boundary(sdc):
    # the largest element count whose workspace fits the scratch passes the size check (it is
    # then refused only because these buffers are far smaller: a pointer error, status 8), and
    # one element more is refused for its size (status 9) -- no kernel runs in either case
    limit = sdc.NOALLOC_SCRATCH_BYTES
    lo, hi = 0, 1 << 40
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if sdc.sdc_grad_average_scan_workspace_size(mid, 4, 2) <= limit:
            lo = mid
        else:
            hi = mid
    assert sdc.sdc_grad_average_scan_workspace_size(lo, 4, 2) <= limit < sdc.sdc_grad_average_scan_workspace_size(
        lo + 1, 4, 2)
    small = [torch.zeros(16, dtype=torch.bfloat16, device=DEV) for _ in range(4)]
    out = torch.empty_like(small[0])
    pre, post = _stats_tensors(4)
    stream = torch.cuda.current_stream().cuda_stream
    for numel, status in ((lo, 8), (lo + 1, 9)):
        with pytest.raises(sdc.SdcError) as ei:
            sdc.sdc_grad_average_scan_noalloc([b.data_ptr() for b in small], out.data_ptr(), numel, 2,
                                              pre.data_ptr(), post.data_ptr(), stream)
        assert ei.value.status == status, (numel, sdc.sdc_last_error())
