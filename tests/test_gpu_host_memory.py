"""Row scans on host memory the GPU reads and writes directly (pinned, or
pageable where the device reads pageable memory), and the refusal of host
pointers by the paths that need device memory."""
import pytest
import torch

import workloads
from checks import assert_rows_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def device_result(mt, x, inclusive):
    d = x.cuda()
    o = torch.empty_like(d)
    mt.mt_scan_rows(d, o, inclusive)
    torch.cuda.synchronize()
    return o.cpu()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("shape", [(1, 1), (3, 33), (5, 4099), (64, 4096), (2, 8192), (3, 12000)],
                         ids=lambda s: f"{s[0]}x{s[1]}")
def test_rows_pinned_host(mt, dtype, inclusive, shape):
    """Pinned host buffers in and out: the kernels read and write them over
    the host link. Same kernel, same bits as the device-memory call, and
    within the oracle tolerance."""
    x = workloads.normal(shape, seed=shape[0] * 31 + shape[1], dtype=dtype).pin_memory()
    out = torch.full(shape, 7.0, dtype=x.dtype).pin_memory()
    mt.mt_scan_rows(x, out, inclusive)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    assert torch.equal(out.view(torch.int16 if x.element_size() == 2 else torch.int32),
                       device_result(mt, x, inclusive).view(torch.int16 if x.element_size() == 2
                                                            else torch.int32))
    assert_rows_close(out, x, dtype, inclusive)


def test_rows_pinned_host_offset_rows(mt):
    """Misaligned row starts inside a pinned buffer, output on the device."""
    base = workloads.normal((7 * 4099 + 3,), seed=5, dtype="bf16").pin_memory()
    x = base[3:].view(7, 4099)
    out = torch.empty((7, 4099), dtype=torch.bfloat16, device="cuda")
    mt.mt_scan_rows(x, out, True)
    torch.cuda.synchronize()
    assert_rows_close(out, x.clone(), "bf16", True)


def test_rows_pageable_host(mt):
    """Plain (pageable) host tensors: scanned in place where the device reads
    pageable memory, refused with MT_ERR_MEMORY elsewhere; never anything else."""
    x = workloads.normal((4, 1000), seed=9, dtype="f32")
    out = torch.full_like(x, 7.0)
    try:
        mt.mt_scan_rows(x, out, False)
    except mt.ScanError as e:
        assert e.code == mt.MT_ERR_MEMORY
        assert torch.all(out == 7.0)
        return
    torch.cuda.synchronize()
    assert_rows_close(out, x, "f32", False)


def test_long_rows_host_refused(mt):
    """Rows longer than one CTA tile use bulk copies: host memory is refused
    and nothing is written."""
    x = workloads.normal((2, 50001), seed=3, dtype="f32").pin_memory()
    out = torch.full_like(x, 7.0).pin_memory()
    with pytest.raises(mt.ScanError) as ei:
        mt.mt_scan_rows(x, out, True)
    assert ei.value.code == mt.MT_ERR_MEMORY
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)


def test_scan1d_and_select_need_device_memory(mt):
    n = 1000
    host = torch.arange(n, dtype=torch.int32).pin_memory()
    dev = host.cuda()
    out = torch.empty_like(dev)
    scr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SCAN)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    with pytest.raises(mt.ScanError) as ei:
        mt.mt_exclusive_scan(host, out, scr, n_dev, "add")
    assert ei.value.code == mt.MT_ERR_MEMORY
    flags = torch.ones(n, dtype=torch.uint8).pin_memory()
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    sscr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
    with pytest.raises(mt.ScanError) as ei:
        mt.mt_select(dev.view(torch.float32), flags, out.view(torch.float32), num, sscr, n_dev)
    assert ei.value.code == mt.MT_ERR_MEMORY
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
