"""Parity of mt_scan_rows_op (product, max, min; CUDA, through the C ABI)
with the CPU oracle."""
import numpy as np
import pytest
import torch

import workloads
from checks import assert_rows_op_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def make(shape, seed, dtype, op):
    if op == "mul":
        return workloads.near_one(shape, seed, dtype)
    return workloads.normal(shape, seed, dtype)


def run(mt, x_cpu, op, inclusive, out_offset=0, inplace=False):
    x = x_cpu.cuda()
    if inplace:
        out = x
    elif out_offset:
        buf = torch.full((x.numel() + out_offset,), 7.0, dtype=x.dtype, device="cuda")
        out = buf[out_offset:].view(x.shape)
    else:
        out = torch.full_like(x, 7.0)
    mt.mt_scan_rows_op(x, out, op, inclusive)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    return out


SHAPES = [(1, 1), (3, 2), (2, 33), (3, 1023), (2, 4096), (5, 4099), (2, 8192), (2, 12289),
          (3, 16385), (2, 50001), (1, 200003)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["mul", "max", "min"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_rows_ops(mt, dtype, op, inclusive, shape):
    x = make(shape, shape[0] * 7 + shape[1], dtype, op)
    out = run(mt, x, op, inclusive)
    assert_rows_op_close(out, x, dtype, op, inclusive)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("op", ["mul", "max", "min", "add"])
def test_rows_ops_misaligned_and_in_place(mt, dtype, op):
    x = make((5, 4099), 101, dtype, op)
    assert_rows_op_close(run(mt, x, op, True, out_offset=3), x, dtype, op, True)
    y = make((3, 30001), 103, dtype, op)
    assert_rows_op_close(run(mt, y, op, False, inplace=True), y, dtype, op, False)


@pytest.mark.parametrize("op", ["max", "min"])
def test_rows_minmax_signed_zero(mt, op):
    """Zero extremes keep the sign of the earliest zero, across tiles of a
    long row and inside a short one."""
    for n in (4096, 100000):
        x = np.full((2, n), 1.0 if op == "min" else -1.0, dtype=np.float32)
        x[0, 17], x[0, n - 5] = -0.0, 0.0
        x[1, 17], x[1, n - 5] = 0.0, -0.0
        t = torch.from_numpy(x)
        for inclusive in (True, False):
            out = run(mt, t, op, inclusive)
            assert_rows_op_close(out, t, "f32", op, inclusive)


def test_rows_op_identities_exclusive(mt):
    """Exclusive out[r][0] is the operation's identity in the storage type."""
    for dtype in ("f32", "bf16", "f16"):
        x = make((4, 100), 5, dtype, "max")
        for op, ident in (("mul", 1.0), ("max", -np.inf), ("min", np.inf), ("add", 0.0)):
            out = run(mt, x, op, False)
            assert torch.all(out[:, 0].float().cpu() == ident), (dtype, op)
