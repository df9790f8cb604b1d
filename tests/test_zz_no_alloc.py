"""mt_scan_rows_noalloc: the row scan for callers that may not allocate.

Programs whose device memory is all reserved up front by another allocator,
that call the scan from a loop where an allocation could take a driver lock
or wait on the device, or whose host forbids device allocations after
start-up, cannot use an entry point that allocates. mt_scan_rows takes the
look-back records of long rows from a memory pool; mt_scan_rows_noalloc uses
a fixed 1 MiB array inside the library instead. These tests check, through
the C ABI, that it gives what mt_scan_rows gives on two calls in a row (the
second reuses the array the first one left behind), and that a shape needing
more than the array is refused before anything is launched.

This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

REL, ABS = 1e-5, 1e-6  # the parity tolerance of the other row-scan tests


def _lib():
    import __graft_entry__
    L = ctypes.CDLL(__graft_entry__._build_module().build())
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mt_scan_rows_noalloc.argtypes = [p, p, i64, i64, i32, i32, p]
    L.mt_scan_rows_noalloc.restype = i32
    return L


def test_noalloc_refuses_too_large_before_launching():
    """Host-side check only: fake, aligned pointers are never touched."""
    L = _lib()
    f32 = 0
    # rows of 8191 tiles of 12288 f32 elements fit (4 header words plus sixteen
    # words per tile); one tile more does not
    assert L.mt_scan_rows_noalloc(0x10000, 0x20000, 1, 8192 * 12288, f32, 1, None) == -7
    assert L.mt_scan_rows_noalloc(0x10000, 0x20000, 2, 4100 * 12288, f32, 0, None) == -7
    assert L.mt_scan_rows_noalloc(0x10000, 0x20000, -1, 5, f32, 1, None) == -1
    assert L.mt_scan_rows_noalloc(0x10000, 0x20000, 0, 5, f32, 1, None) == 0


def _bound(x_cpu, ref, dtype):
    mag = torch.cumsum(x_cpu.double().abs(), dim=-1).numpy()
    bound = REL * mag + ABS
    if dtype != "f32":
        import oracle
        bound = bound + oracle.ulp_array(ref, dtype)
    return bound


@pytest.mark.gpu
def test_noalloc_matches_scan_rows_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    import prefix_scan_row_gb300 as mt
    cases = [("f32", workloads.rows_long(rows=4, n=1 << 20), True),
             ("bf16", workloads.rows_half(3, 300001, "bf16"), False)]
    xs = [c[1].cuda() for c in cases]
    got = [torch.full_like(x, 9.0) for x in xs]
    want = [torch.full_like(x, -9.0) for x in xs]
    # two no-allocation calls back to back on one stream, then the ordinary ones
    for (_, _, inclusive), x, g in zip(cases, xs, got):
        mt.mt_scan_rows_noalloc(x, g, inclusive)
    for (_, _, inclusive), x, w in zip(cases, xs, want):
        mt.mt_scan_rows(x, w, inclusive)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    for (dtype, x_cpu, _), g, w in zip(cases, got, want):
        g64 = g.cpu().double().numpy()
        w64 = w.cpu().double().numpy()
        bound = _bound(x_cpu, w64, dtype)
        bad = np.nonzero(~(np.abs(g64 - w64) <= bound))
        assert bad[0].size == 0, f"{dtype}: {bad[0].size} elements differ beyond the tolerance"
