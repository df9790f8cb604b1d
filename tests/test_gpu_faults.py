"""Failure detection of the look-back without faulting the GPU.

A host-side test hook makes one tile skip publishing its status ("a flag that
nothing sets"). The tiles after it wait a bounded number of polls, give up,
record MT_ERR_LOOKBACK_TIMEOUT in the device error word and let the kernel
finish; mt_scan_status() reports it, and the next call on the same context
is correct again.
"""
import numpy as np
import pytest
import torch

import oracle
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


@pytest.mark.parametrize("dtype", ["i64", "f64"])
def test_scan_8byte_timeout_reported_then_recovers(mt, dtype):
    """8-byte status records (i64), and the per-thread-run form that f64
    tiles take, whose warp 0 looks back on its own."""
    n = 1 << 20
    if dtype == "i64":
        arr_cpu = workloads.randint((n,), 4, 0, 1 << 20, "i64")
    else:
        arr_cpu = workloads.uniform64((n,), 4, -1.0, 1.0)
    arr = arr_cpu.cuda()
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=3, spin_limit=4096)
        _scan(mt, arr, n)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    out = _scan(mt, arr, n)
    assert mt.mt_scan_status() == 0
    assert_scan_matches(out, arr_cpu, n, dtype, "add")


def test_select_wide_timeout_reported_then_recovers(mt):
    n = 1 << 20
    vals, flags = workloads.select_inputs(n, 0.5, seed=10)
    arr, fl = vals.to(torch.float64).cuda(), flags.cuda()
    out = torch.empty_like(arr)
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=2, spin_limit=4096)
        mt.mt_select_wide(arr, fl, out, num, scratch, n_dev)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    mt.mt_select_wide(arr, fl, out, num, scratch, n_dev)
    assert mt.mt_scan_status() == 0
    k = int(num.item())
    want = vals.to(torch.float64)[flags.bool()]
    assert k == want.numel()
    assert torch.equal(out[:k].cpu().view(torch.int64), want.view(torch.int64))


@pytest.mark.parametrize("words", [3, 5])
def test_select_struct_timeout_reported_then_recovers(mt, words):
    """Struct elements (flags staged, values read after the look-back), with
    W known at compile time (3) and at run time (5)."""
    n = 1 << 20
    vals = workloads.randint((n, words), 11, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(n, 0.5, 12)
    arr, fl = vals.cuda(), flags.cuda()
    out = torch.empty_like(arr)
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=2, spin_limit=4096)
        mt.mt_select_wide(arr, fl, out, num, scratch, n_dev)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    mt.mt_select_wide(arr, fl, out, num, scratch, n_dev)
    assert mt.mt_scan_status() == 0
    k = int(num.item())
    want = vals[flags.bool()]
    assert k == want.shape[0]
    assert torch.equal(out[:k].cpu(), want)


def test_reduce_by_key_timeout_reported_then_recovers(mt):
    n = 1 << 20
    keys, vals = workloads.runs(n, 8.0, 11, "i32", "i32")
    k, v = keys.cuda(), vals.cuda()
    ko, vo = torch.empty_like(k), torch.empty_like(v)
    nr = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_REDUCE_BY_KEY)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=4, spin_limit=4096)
        mt.mt_reduce_by_key_add(k, v, ko, vo, nr, scratch, n_dev)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    mt.mt_reduce_by_key_add(k, v, ko, vo, nr, scratch, n_dev)
    assert mt.mt_scan_status() == 0
    want_k, want_v, r = oracle.reduce_by_key_add(keys, vals, n, "i32", "i32")
    assert int(nr.item()) == r
    assert np.array_equal(ko[:r].cpu().numpy(), want_k) and np.array_equal(vo[:r].cpu().numpy(), want_v)
