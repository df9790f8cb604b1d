"""mt_scan_rows_noalloc: the row scan for callers that may not allocate.

Some programs cannot let a library allocate device memory: their memory is
all reserved up front by another allocator (a framework's caching allocator,
a fixed arena), they call the scan from a loop where an allocation could take
a driver lock or wait on the device, or their host forbids allocations after
start-up. mt_scan_rows takes the look-back records of long rows from a
memory pool; mt_scan_rows_noalloc uses a fixed 1 MiB array inside the
library instead.

These tests check, through the C ABI, that it computes the row scan (against
the CPU oracle, exactly on inputs whose every partial sum is exact, and
against mt_scan_rows) on two calls in a row (the second reuses the array the
first left behind), that a look-back wait that gives up is reported and the
next call is correct, that calls allocate no device memory, and that a shape
needing more than the array is refused before anything is launched.

The file name sorts last so that pytest collects it after every other test
file: if it fails, a run that stops at the first failure has already run
everything else.
"""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import workloads
from checks import assert_rows_close

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REL, ABS = 1e-5, 1e-6  # the parity tolerance of the other row-scan tests
F32, BF16, TOO_LARGE = 0, 1, -7


def _lib():
    import __graft_entry__
    L = ctypes.CDLL(__graft_entry__._build_module().build())
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mt_scan_rows_noalloc.argtypes = [p, p, i64, i64, i32, i32, p]
    L.mt_scan_rows_noalloc.restype = i32
    L.mt_scan_rows_scratch_slots.argtypes = [i64, i64, i32]
    L.mt_scan_rows_scratch_slots.restype = i64
    return L


def _largest_fitting_n(L, rows, dtype, limit_bytes):
    """The largest row length whose workspace, as the library sizes it, fits."""
    lo, hi = 1, 1 << 36
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if L.mt_scan_rows_scratch_slots(rows, mid, dtype) * 8 <= limit_bytes:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_refuses_too_large_before_launching():
    """Host-side checks only: the fake pointers are never dereferenced (a
    refused call returns before any CUDA call; a call that fits fails later,
    on the pointer check or, without a GPU, on the device query)."""
    L = _lib()
    limit = 1 << 20  # MT_NOALLOC_SCRATCH_BYTES
    # misaligned row starts, so that the call's plan is the worst case the
    # sizing call reports
    for rows, dtype, inp, out in ((1, F32, 0x10004, 0x20004), (3, F32, 0x10004, 0x20004),
                                  (2, BF16, 0x10002, 0x20002)):
        n = _largest_fitting_n(L, rows, dtype, limit)
        assert L.mt_scan_rows_scratch_slots(rows, n, dtype) > 0
        assert L.mt_scan_rows_noalloc(inp, out, rows, n + 1, dtype, 1, None) == TOO_LARGE
        assert L.mt_scan_rows_noalloc(inp, out, rows, n, dtype, 0, None) != TOO_LARGE
    assert L.mt_scan_rows_noalloc(0x10000, 0x20000, -1, 5, F32, 1, None) == -1
    assert L.mt_scan_rows_noalloc(0x10000, 0x20000, 0, 5, F32, 1, None) == 0


def _within(got, want, x_cpu, dtype):
    """got within the parity tolerance of want (both device tensors)."""
    g64 = got.cpu().double().numpy()
    w64 = want.cpu().double().numpy()
    bound = REL * torch.cumsum(x_cpu.double().abs(), dim=-1).numpy() + ABS
    if dtype != "f32":
        import oracle
        bound = bound + oracle.ulp_array(w64, dtype)
    return int(np.count_nonzero(~(np.abs(g64 - w64) <= bound)))


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import prefix_scan_row_gb300 as mt
    # (dtype, input, inclusive, exact): long rows of several tiles each
    cases = [("f32", workloads.rows_long(rows=4, n=1 << 20), True, False),
             ("bf16", workloads.rows_half(3, 300001, "bf16"), False, False),
             ("f32", workloads.dyadic((2, (1 << 19) + 5), 31, "f32"), False, True),
             ("f16", workloads.dyadic((3, 70001), 32, "f16"), True, True)]
    xs = [c[1].cuda() for c in cases]
    for x in xs:
        assert mt.mt_scan_rows_scratch_slots(x.shape[0], x.shape[1], x.dtype) > 0  # the array is used
    firsts = [torch.full_like(x, 9.0) for x in xs]
    seconds = [torch.full_like(x, 7.0) for x in xs]
    want = [torch.full_like(x, -9.0) for x in xs]
    # every case twice, back to back on one stream: each call clears and reuses
    # what the one before left in the shared array
    for (_, _, inclusive, _), x, a, b in zip(cases, xs, firsts, seconds):
        mt.mt_scan_rows_noalloc(x, a, inclusive)
        mt.mt_scan_rows_noalloc(x, b, inclusive)
    for (_, _, inclusive, _), x, w in zip(cases, xs, want):
        mt.mt_scan_rows(x, w, inclusive)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    for (dtype, x_cpu, inclusive, exact), a, b, w in zip(cases, firsts, seconds, want):
        for got in (a, b):
            assert_rows_close(got, x_cpu, dtype, inclusive, exact=exact)
            bad = _within(got, w, x_cpu, dtype)
            assert bad == 0, f"{dtype}: {bad} elements differ from mt_scan_rows beyond the tolerance"


@pytest.mark.gpu
def test_noalloc_timeout_reported_then_recovers():
    """The look-back test hook applies: a tile that never publishes makes its
    successors give up; the error is reported and the next call is right."""
    import prefix_scan_row_gb300 as mt
    x_cpu = workloads.rows_long(rows=2, n=1 << 18)
    x = x_cpu.cuda()
    out = torch.empty_like(x)
    assert mt.mt_scan_status() == 0
    try:
        mt.mt_scan_debug_lookback(skip_publish_tile=2, spin_limit=4096)
        mt.mt_scan_rows_noalloc(x, out, True)
        assert mt.mt_scan_status() == mt.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        mt.mt_scan_debug_lookback(-1, 0)
    mt.mt_scan_rows_noalloc(x, out, True)
    assert mt.mt_scan_status() == 0
    assert_rows_close(out, x_cpu, "f32", True)


_NO_ALLOC_CHILD = r"""
import json, sys, torch
sys.path.insert(0, sys.argv[1])
import prefix_scan_row_gb300 as mt
import workloads
torch.cuda.set_device(0)
xs = [workloads.rows_long(rows=4, n=1 << 20).cuda(), workloads.rows_half(3, 300001, "bf16").cuda()]
outs = [torch.empty_like(x) for x in xs]
def calls():
    for x, o in zip(xs, outs):
        mt.mt_scan_rows_noalloc(x, o, True)
calls()  # loads the kernels and finds the array's address
torch.cuda.synchronize()
before = torch.cuda.mem_get_info()[0]
for _ in range(5):
    calls()
torch.cuda.synchronize()
after = torch.cuda.mem_get_info()[0]
print(json.dumps({"before": before, "after": after, "status": mt.mt_scan_status()}))
"""


@pytest.mark.gpu
def test_noalloc_allocates_nothing():
    """In a fresh process (the library's pool never created), the free device
    memory is the same before and after a series of long-row calls."""
    r = subprocess.run([sys.executable, "-c", _NO_ALLOC_CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    got = json.loads(r.stdout.strip().splitlines()[-1])
    assert got["status"] == 0
    assert got["after"] == got["before"], f"free device memory changed: {got}"
