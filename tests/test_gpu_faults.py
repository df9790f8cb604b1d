"""Failure detection of the look-back without faulting the GPU.

A host-side test hook makes one tile skip publishing its status ("a flag that
nothing sets"). The tiles after it wait a bounded number of polls, give up,
record MT_ERR_LOOKBACK_TIMEOUT in the device error word and let the kernel
finish; mt_scan_status() reports it, and the next call on the same context
is correct again.
"""
import pytest
import torch

import workloads
from checks import assert_rows_close, assert_scan_matches, assert_select_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def _scan(mt, arr, n):
    out = torch.zeros_like(arr)
    scratch = mt.alloc_scratch(arr.numel(), arr.dtype, mt.MT_SCRATCH_SCAN)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_exclusive_scan(arr, out, scratch, n_dev, "add")
    return out


def test_scan_timeout_reported_then_recovers(mt):
    n = 1 << 20
    arr_cpu = workloads.randint((n,), 3, 0, 16, "i32")
    arr = arr_cpu.cuda()
    assert mt.mt_scan_status() == 0
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=5, spin_limit=4096)
        _scan(mt, arr, n)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    assert mt.mt_scan_status() == 0  # the word was cleared by the read
    out = _scan(mt, arr, n)
    assert mt.mt_scan_status() == 0
    assert_scan_matches(out, arr_cpu, n, "i32", "add")


def test_rows_timeout_reported_then_recovers(mt):
    x_cpu = workloads.rows_long(rows=2, n=1 << 18)
    x = x_cpu.cuda()
    out = torch.empty_like(x)
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=2, spin_limit=4096)
        mt.mt_scan_rows(x, out, True)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    mt.mt_scan_rows(x, out, True)
    assert mt.mt_scan_status() == 0
    assert_rows_close(out, x_cpu, "f32", True)


def test_select_timeout_reported_then_recovers(mt):
    n = 1 << 20
    vals, flags = workloads.select_inputs(n, 0.5, seed=9)
    arr, fl = vals.cuda(), flags.cuda()
    out = torch.empty_like(arr)
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=1, spin_limit=4096)
        mt.mt_select(arr, fl, out, num, scratch, n_dev)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    mt.mt_select(arr, fl, out, num, scratch, n_dev)
    assert mt.mt_scan_status() == 0
    assert_select_matches(out, num, vals, flags, n)
