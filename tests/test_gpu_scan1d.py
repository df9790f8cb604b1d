"""Parity of mt_exclusive_scan (CUDA, through the C ABI) with the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from checks import assert_scan_matches

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


def run_scan(mt, arr_cpu, n, dtype, op, arr_off=0, out_off=0, scratch_cap=None):
    cap = arr_cpu.numel()
    abuf = torch.zeros(cap + arr_off, dtype=TDT[dtype], device="cuda")
    arr = abuf[arr_off:]
    arr.copy_(arr_cpu.cuda())
    obuf = torch.full((cap + out_off + 16,), SENTINEL[dtype], dtype=TDT[dtype], device="cuda")
    out = obuf[out_off:out_off + cap]
    scratch = mt.alloc_scratch(scratch_cap or max(cap, 1), TDT[dtype], mt.MT_SCRATCH_SCAN)
    scratch.fill_(-1)  # garbage: the call needs no initialised scratch
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_exclusive_scan(arr, out, scratch, n_dev, op)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    # everything past n (and the guard band) keeps its sentinel
    assert torch.all(obuf[out_off + max(n, 0):] == SENTINEL[dtype]).item()
    if out_off:
        assert torch.all(obuf[:out_off] == SENTINEL[dtype]).item()
    return out


SIZES = [0, 1, 2, 3, 5, 31, 33, 1023, 4095, 4096, 4097, 8191, 8193, 12345, 100003, (1 << 20) + 7]


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("n", SIZES)
def test_scan_sizes(mt, dtype, op, n):
    cap = n + 37  # live count below the capacity
    arr = make_input(dtype, cap, seed=n + 1)
    out = run_scan(mt, arr, n, dtype, op)
    assert_scan_matches(out, arr, n, dtype, op)


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("op", ["add", "max"])
@pytest.mark.parametrize("offs", [(1, 0), (0, 1), (1, 1), (3, 2)])
def test_scan_misaligned(mt, dtype, op, offs):
    n = 50001
    arr = make_input(dtype, n + 5, seed=77)
    out = run_scan(mt, arr, n, dtype, op, arr_off=offs[0], out_off=offs[1], scratch_cap=n + 5)
    assert_scan_matches(out, arr, n, dtype, op)


def test_scan_i32_wraps(mt):
    n = 300000
    arr = workloads.randint((n,), 5, 1 << 28, 1 << 30, "i32")  # the sum passes 2^31 many times
    out = run_scan(mt, arr, n, "i32", "add")
    assert_scan_matches(out, arr, n, "i32", "add")


def test_scan_i64_wraps(mt):
    n = 100000
    arr = workloads.randint((n,), 6, 1 << 58, 1 << 62, "i64")
    out = run_scan(mt, arr, n, "i64", "add")
    assert_scan_matches(out, arr, n, "i64", "add")


@pytest.mark.parametrize("op", ["min", "max"])
def test_scan_f32_infinities(mt, op):
    n = 70000
    arr = workloads.uniform((n,), 8, -1.0, 1.0, "f32")
    arr[[5, 4100, 9000, 65000]] = torch.tensor([np.inf, -np.inf, np.inf, -np.inf])
    out = run_scan(mt, arr, n, "f32", op)
    assert_scan_matches(out, arr, n, "f32", op)


def test_scan_f32_add_dyadic_exact(mt):
    n = 1 << 15
    arr = workloads.dyadic((n,), 12, "f32")
    out = run_scan(mt, arr, n, "f32", "add")
    ref = oracle.exclusive_scan(arr, n, "f32", "add")
    assert np.array_equal(out[:n].cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_scan_negative_count_is_empty(mt):
    arr = make_input("i32", 100, 1)
    out = run_scan(mt, arr, -5, "i32", "add", scratch_cap=100)
    assert torch.all(out == SENTINEL["i32"]).item()


def test_scan_reuses_dirty_scratch(mt):
    """Back-to-back calls on one scratch buffer with different counts."""
    cap = 200000
    arr_cpu = make_input("i32", cap, 4)
    arr = arr_cpu.cuda()
    scratch = mt.alloc_scratch(cap, torch.int32, mt.MT_SCRATCH_SCAN)
    for n in (cap, 12345, cap - 1, 4097):
        out = torch.zeros(cap, dtype=torch.int32, device="cuda")
        n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
        mt.mt_exclusive_scan(arr, out, scratch, n_dev, "add")
        torch.cuda.synchronize()
        assert_scan_matches(out, arr_cpu, n, "i32", "add")


# ---- the configured workload at full size ----------------------------------

@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
def test_scan_full_size(mt, dtype):
    cap, n = workloads.SCAN1D_CAPACITY, workloads.SCAN1D_LIVE
    arr_cpu = workloads.scan1d(dtype)
    arr = arr_cpu.cuda()
    scratch = mt.alloc_scratch(cap, TDT[dtype], mt.MT_SCRATCH_SCAN)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    out = torch.empty(cap, dtype=TDT[dtype], device="cuda")
    for op in ("add", "min", "max"):
        out.fill_(SENTINEL[dtype])
        mt.mt_exclusive_scan(arr, out, scratch, n_dev, op)
        torch.cuda.synchronize()
        assert mt.mt_scan_status() == 0
        assert torch.all(out[n:] == SENTINEL[dtype]).item()
        assert_scan_matches(out, arr_cpu, n, dtype, op)


@pytest.mark.parametrize("op", ["min", "max"])
def test_scan_f32_signed_zeros_bit_exact(mt, op):
    """Both zeros present: which one a min/max keeps depends on element order
    (the earlier one wins), so tiles whose extreme is a zero must combine in
    order. Bit-exact against the oracle."""
    n = 300001
    u = workloads.uniform((n,), 21, 0.0, 1.0, "f32")
    arr = u if op == "min" else -u
    g = torch.Generator().manual_seed(22)
    pos = torch.randperm(n, generator=g)[:400]
    arr[pos[:200]] = 0.0
    arr[pos[200:]] = -0.0
    out = run_scan(mt, arr, n, "f32", op)
    assert_scan_matches(out, arr, n, "f32", op)
