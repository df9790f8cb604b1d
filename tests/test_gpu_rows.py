"""Parity of mt_scan_rows (CUDA, through the C ABI) with the CPU oracle."""
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


def run_rows(mt, x_cpu, inclusive, inplace=False, out_offset=0):
    x = x_cpu.cuda()
    if inplace:
        out = x
    elif out_offset:
        buf = torch.full((x.numel() + out_offset,), 7.0, dtype=x.dtype, device="cuda")
        out = buf[out_offset:].view(x.shape)
    else:
        out = torch.full_like(x, 7.0)
    mt.mt_scan_rows(x, out, inclusive)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    return out


SHAPES = [(1, 1), (3, 2), (2, 3), (5, 4), (2, 5), (4, 7), (3, 8), (2, 31), (2, 32), (3, 33),
          (2, 255), (2, 256), (2, 257), (3, 1023), (2, 1024), (2, 1025), (2, 2047), (2, 2049),
          (3, 4095), (2, 4096), (3, 4097), (2, 8191), (2, 8192), (2, 8193), (5, 4099),
          (2, 16385), (3, 50001), (1, 200003), (9, 3)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_rows_shapes(mt, dtype, inclusive, shape):
    x = workloads.normal(shape, seed=shape[0] * 7919 + shape[1], dtype=dtype)
    out = run_rows(mt, x, inclusive)
    assert_rows_close(out, x, dtype, inclusive)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("shape", [(3, 1000), (4, 4099), (2, 8192), (3, 20001), (2, 1 << 15)])
def test_rows_dyadic_bit_exact(mt, dtype, inclusive, shape):
    """k/256 inputs: every partial sum is exact in f32, so any grouping gives
    the oracle's bits."""
    x = workloads.dyadic(shape, seed=11 + shape[1], dtype=dtype)
    out = run_rows(mt, x, inclusive)
    assert_rows_close(out, x, dtype, inclusive, exact=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(5, 4099), (3, 30001), (2, 8192)])
def test_rows_in_place(mt, dtype, shape):
    x = workloads.normal(shape, seed=3, dtype=dtype)
    out = run_rows(mt, x, True, inplace=True)
    assert_rows_close(out, x, dtype, True)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("off", [1, 3])
@pytest.mark.parametrize("shape", [(4, 1000), (3, 4099), (2, 30001)])
def test_rows_output_other_alignment(mt, dtype, off, shape):
    """Output rows with a different 16-byte phase from the input rows."""
    x = workloads.normal(shape, seed=5, dtype=dtype)
    out = run_rows(mt, x, False, out_offset=off)
    assert_rows_close(out, x, dtype, False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rows_input_misaligned_start(mt, dtype):
    """Tensor starting one element past a 16-byte boundary."""
    x_cpu = workloads.normal((6, 3001), seed=9, dtype=dtype)
    big = torch.zeros(x_cpu.numel() + 1, dtype=x_cpu.dtype, device="cuda")
    x = big[1:].view(x_cpu.shape)
    x.copy_(x_cpu.cuda())
    out = torch.zeros_like(x)
    mt.mt_scan_rows(x, out, True)
    torch.cuda.synchronize()
    assert_rows_close(out, x_cpu, dtype, True)


def test_rows_empty_is_noop(mt):
    for shape in [(0, 5), (4, 0)]:
        x = torch.zeros(shape, device="cuda")
        out = torch.zeros(shape, device="cuda")
        mt.mt_scan_rows(x, out, True)
    torch.cuda.synchronize()


def test_rows_guard_band_untouched(mt):
    """Elements after the tensor keep their sentinel."""
    x_cpu = workloads.normal((3, 4099), seed=2, dtype="bf16")
    buf = torch.full((x_cpu.numel() + 64,), 123.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:x_cpu.numel()].view(x_cpu.shape)
    mt.mt_scan_rows(x_cpu.cuda(), out, False)
    torch.cuda.synchronize()
    assert torch.all(buf[x_cpu.numel():] == 123.0)
    assert_rows_close(out, x_cpu, "bf16", False)


# ---- the configured workloads at full size --------------------------------

@pytest.mark.parametrize("inclusive", [True, False])
def test_rows_f32_1024x4096(mt, inclusive):
    x = workloads.rows_f32()
    assert_rows_close(run_rows(mt, x, inclusive), x, "f32", inclusive)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rows_half_8192x8192_exclusive(mt, dtype):
    x = workloads.rows_half(8192, 8192, dtype)
    assert_rows_close(run_rows(mt, x, False), x, dtype, False)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rows_half_4096x4099_inclusive(mt, dtype):
    x = workloads.rows_half(4096, 4099, dtype)
    assert_rows_close(run_rows(mt, x, True), x, dtype, True)


@pytest.mark.parametrize("inclusive", [True, False])
def test_rows_long_4x2pow24(mt, inclusive):
    x = workloads.rows_long()
    assert_rows_close(run_rows(mt, x, inclusive), x, "f32", inclusive)
