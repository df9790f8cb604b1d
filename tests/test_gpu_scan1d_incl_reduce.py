"""Parity of mt_inclusive_scan and mt_reduce (CUDA, through the C ABI) with
the CPU oracle."""
import numpy as np
import pytest
import torch

import workloads
from checks import assert_reduce_matches, assert_scan_matches

pytestmark = pytest.mark.gpu

TDT = {"i32": torch.int32, "i64": torch.int64, "f32": torch.float32}
SENTINEL = {"i32": -123456789, "i64": -1234567890123, "f32": -777.25}


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def make_input(dtype, cap, seed):
    if dtype == "i32":
        return workloads.randint((cap,), seed, -1000, 1000, "i32")
    if dtype == "i64":
        return workloads.randint((cap,), seed, -(1 << 40), 1 << 40, "i64")
    return workloads.uniform((cap,), seed, -1.0, 1.0, "f32")


def run_inclusive(mt, arr_cpu, n, dtype, op, arr_off=0, out_off=0, inplace=False):
    cap = arr_cpu.numel()
    abuf = torch.zeros(cap + arr_off + 16, dtype=TDT[dtype], device="cuda")
    arr = abuf[arr_off:arr_off + cap]
    arr.copy_(arr_cpu.cuda())
    if inplace:
        obuf, out = abuf, arr
    else:
        obuf = torch.full((cap + out_off + 16,), SENTINEL[dtype], dtype=TDT[dtype], device="cuda")
        out = obuf[out_off:out_off + cap]
    scratch = mt.alloc_scratch(max(cap, 1), TDT[dtype], mt.MT_SCRATCH_SCAN)
    scratch.fill_(-1)  # garbage: the call needs no initialised scratch
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_inclusive_scan(arr, out, scratch, n_dev, op)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    if not inplace:
        assert torch.all(obuf[out_off + max(n, 0):] == SENTINEL[dtype]).item()
        if out_off:
            assert torch.all(obuf[:out_off] == SENTINEL[dtype]).item()
    else:  # past n the input is untouched
        assert torch.equal(arr[max(n, 0):].cpu(), arr_cpu[max(n, 0):])
    return out


def run_reduce(mt, arr_cpu, n, dtype, op, arr_off=0):
    cap = arr_cpu.numel()
    abuf = torch.zeros(cap + arr_off + 16, dtype=TDT[dtype], device="cuda")
    arr = abuf[arr_off:arr_off + cap]
    arr.copy_(arr_cpu.cuda())
    out = torch.full((3,), SENTINEL[dtype], dtype=TDT[dtype], device="cuda")
    scratch = mt.alloc_scratch(cap, TDT[dtype], mt.MT_SCRATCH_REDUCE)
    scratch.fill_(-1)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_reduce(arr, out, scratch, n_dev, op)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    assert torch.all(out[1:] == SENTINEL[dtype]).item()
    return out


SIZES = [0, 1, 2, 3, 5, 31, 33, 4097, 12287, 12288, 12289, 100003, (1 << 20) + 7]


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("n", SIZES)
def test_inclusive_sizes(mt, dtype, op, n):
    arr = make_input(dtype, n + 37, seed=n + 3)
    out = run_inclusive(mt, arr, n, dtype, op)
    assert_scan_matches(out, arr, n, dtype, op, inclusive=True)


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("offs", [(1, 0), (0, 1), (3, 2)])
def test_inclusive_misaligned(mt, dtype, offs):
    n = 50001
    arr = make_input(dtype, n + 5, seed=79)
    out = run_inclusive(mt, arr, n, dtype, "add", arr_off=offs[0], out_off=offs[1])
    assert_scan_matches(out, arr, n, dtype, "add", inclusive=True)


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("off", [0, 1])
@pytest.mark.parametrize("op", ["add", "max"])
def test_inclusive_in_place(mt, dtype, off, op):
    n = 200001
    arr = make_input(dtype, n + 9, seed=81)
    out = run_inclusive(mt, arr, n, dtype, op, arr_off=off, inplace=True)
    assert_scan_matches(out, arr, n, dtype, op, inclusive=True)


def test_inclusive_i32_wraps(mt):
    n = 300000
    arr = workloads.randint((n,), 6, 1 << 28, 1 << 30, "i32")
    out = run_inclusive(mt, arr, n, "i32", "add")
    assert_scan_matches(out, arr, n, "i32", "add", inclusive=True)


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("n", SIZES + [3_000_017])
def test_reduce_sizes(mt, dtype, op, n):
    arr = make_input(dtype, n + 37, seed=n + 5)
    out = run_reduce(mt, arr, n, dtype, op)
    assert_reduce_matches(out, arr, n, dtype, op)


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("off", [1, 2, 3])
@pytest.mark.parametrize("op", ["add", "min"])
def test_reduce_misaligned(mt, dtype, off, op):
    n = 77777
    arr = make_input(dtype, n, seed=83)
    out = run_reduce(mt, arr, n, dtype, op, arr_off=off)
    assert_reduce_matches(out, arr, n, dtype, op)


def test_reduce_i32_wraps(mt):
    n = 1_000_003
    arr = workloads.randint((n,), 7, 1 << 28, 1 << 30, "i32")
    out = run_reduce(mt, arr, n, "i32", "add")
    assert_reduce_matches(out, arr, n, "i32", "add")


@pytest.mark.parametrize("first_negative", [False, True])
def test_f32_min_max_signed_zero(mt, first_negative):
    """Zero extremes keep the sign of the earliest zero, whatever CTA holds it."""
    n = 3_000_000
    x = np.ones(n, dtype=np.float32)
    y = -np.ones(n, dtype=np.float32)
    i, j = 1_234_567, 2_500_001  # the two zeros, in different tiles and CTAs
    a, b = (np.float32(-0.0), np.float32(0.0)) if first_negative else (np.float32(0.0), np.float32(-0.0))
    x[i], x[j] = a, b
    y[i], y[j] = a, b
    for arr, op in ((x, "min"), (y, "max")):
        t = torch.from_numpy(arr)
        out = run_reduce(mt, t, n, "f32", op)
        assert_reduce_matches(out, t, n, "f32", op)
        assert np.signbit(out[0].item()) == first_negative
        inc = run_inclusive(mt, t, n, "f32", op)
        assert_scan_matches(inc, t, n, "f32", op, inclusive=True)


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
def test_full_size_config(mt, dtype):
    """The configured 1-D workload: capacity 2^28, live n = 2^28 - 12345."""
    cap, n = workloads.SCAN1D_CAPACITY, workloads.SCAN1D_LIVE
    arr = workloads.scan1d(dtype, capacity=cap)
    for op in ("add", "min", "max"):
        out = run_reduce(mt, arr, n, dtype, op)
        assert_reduce_matches(out, arr, n, dtype, op)
    out = run_inclusive(mt, arr, n, dtype, "add")
    assert_scan_matches(out, arr, n, dtype, "add", inclusive=True)
