"""Parity of the 1-D scans and the reduce for u32, u64 and f64 (CUDA, through
the C ABI) with the CPU oracle. Unsigned buffers are allocated through their
signed twins and viewed as unsigned, so only view operations touch them."""
import numpy as np
import pytest
import torch

import workloads
from checks import assert_reduce_matches, assert_scan_matches

pytestmark = pytest.mark.gpu

TDT = {"u32": torch.uint32, "u64": torch.uint64, "f64": torch.float64}
TWIN = {"u32": torch.int32, "u64": torch.int64, "f64": torch.float64}
SENT = {"u32": -123456789, "u64": -1234567890123, "f64": -777.25}


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def make_input(dtype, cap, seed):
    if dtype == "f64":
        return workloads.uniform64((cap,), seed, -1.0, 1.0)
    return workloads.bits_uniform((cap,), seed, dtype)


def to_twin(t):
    return t.view({torch.uint32: torch.int32, torch.uint64: torch.int64}.get(t.dtype, t.dtype))


def dev_copy(dtype, x_cpu, off=0, extra=16):
    buf = torch.zeros(x_cpu.numel() + off + extra, dtype=TWIN[dtype], device="cuda")
    buf[off:off + x_cpu.numel()].copy_(to_twin(x_cpu).cuda())
    return buf, buf[off:off + x_cpu.numel()].view(TDT[dtype])


def run_scan(mt, x_cpu, n, dtype, op, inclusive, arr_off=0, out_off=0):
    cap = x_cpu.numel()
    _, arr = dev_copy(dtype, x_cpu, arr_off)
    obuf = torch.full((cap + out_off + 16,), SENT[dtype], dtype=TWIN[dtype], device="cuda")
    out = obuf[out_off:out_off + cap].view(TDT[dtype])
    scr = mt.alloc_scratch(max(cap, 1), TDT[dtype], mt.MT_SCRATCH_SCAN)
    scr.fill_(-1)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    (mt.mt_inclusive_scan if inclusive else mt.mt_exclusive_scan)(arr, out, scr, n_dev, op)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    assert torch.all(obuf[out_off + max(n, 0):] == SENT[dtype]).item()
    return out


def run_reduce(mt, x_cpu, n, dtype, op, arr_off=0):
    _, arr = dev_copy(dtype, x_cpu, arr_off)
    obuf = torch.full((3,), SENT[dtype], dtype=TWIN[dtype], device="cuda")
    out = obuf.view(TDT[dtype])
    scr = mt.alloc_scratch(x_cpu.numel(), TDT[dtype], mt.MT_SCRATCH_REDUCE)
    scr.fill_(-1)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_reduce(arr, out, scr, n_dev, op)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    assert torch.all(obuf[1:] == SENT[dtype]).item()
    return out


SIZES = [0, 1, 5, 33, 6143, 6145, 12289, 100003, (1 << 20) + 7]


@pytest.mark.parametrize("dtype", ["u32", "u64", "f64"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("inclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_scan_ext(mt, dtype, op, inclusive, n):
    x = make_input(dtype, n + 11, seed=n + 13)
    out = run_scan(mt, x, n, dtype, op, inclusive)
    assert_scan_matches(out, x, n, dtype, op, inclusive=inclusive)


@pytest.mark.parametrize("dtype", ["u32", "u64", "f64"])
@pytest.mark.parametrize("offs", [(1, 0), (0, 1), (3, 2)])
def test_scan_ext_misaligned(mt, dtype, offs):
    n = 50001
    x = make_input(dtype, n + 5, seed=89)
    for op in ("add", "max"):
        out = run_scan(mt, x, n, dtype, op, False, arr_off=offs[0], out_off=offs[1])
        assert_scan_matches(out, x, n, dtype, op)


@pytest.mark.parametrize("dtype", ["u32", "u64", "f64"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("n", SIZES + [3_000_017])
def test_reduce_ext(mt, dtype, op, n):
    x = make_input(dtype, n + 11, seed=n + 17)
    out = run_reduce(mt, x, n, dtype, op)
    assert_reduce_matches(out, x, n, dtype, op)


def test_unsigned_order_across_tiles(mt):
    """The largest values have the top bit set: a signed comparison would
    pick the wrong extremes."""
    n = 1_000_003
    x = np.full(n, 5, dtype=np.uint32)
    x[777_777] = 2**32 - 2
    x[123] = 1
    t = torch.from_numpy(x.view(np.int32).copy()).view(torch.uint32)
    for op in ("min", "max"):
        assert_reduce_matches(run_reduce(mt, t, n, "u32", op), t, n, "u32", op)
        assert_scan_matches(run_scan(mt, t, n, "u32", op, True), t, n, "u32", op, inclusive=True)
    y = np.full(n, 5, dtype=np.uint64)
    y[654_321] = 2**64 - 3
    u = torch.from_numpy(y.view(np.int64).copy()).view(torch.uint64)
    assert_reduce_matches(run_reduce(mt, u, n, "u64", "max"), u, n, "u64", "max")
    assert_scan_matches(run_scan(mt, u, n, "u64", "add", False), u, n, "u64", "add")


@pytest.mark.parametrize("first_negative", [False, True])
def test_f64_min_max_signed_zero(mt, first_negative):
    n = 3_000_000
    a, b = (-0.0, 0.0) if first_negative else (0.0, -0.0)
    for op, fill in (("min", 1.0), ("max", -1.0)):
        x = np.full(n, fill)
        x[1_111_111], x[2_900_001] = a, b
        t = torch.from_numpy(x)
        out = run_reduce(mt, t, n, "f64", op)
        assert_reduce_matches(out, t, n, "f64", op)
        assert np.signbit(out[0].item()) == first_negative
        assert_scan_matches(run_scan(mt, t, n, "f64", op, True), t, n, "f64", op, inclusive=True)


@pytest.mark.parametrize("seed", [11, 12])
def test_f64_min_max_special_values(mt, seed):
    """f64 min/max over infinities, subnormals, both zeros, values one ulp
    apart and the extreme finite values: every combine order the kernels use
    must give the serial result bit for bit. Inputs are NaN-free."""
    tiny, mn, big = 5e-324, 2.2250738585072014e-308, 1.7976931348623157e308
    pool = np.array([np.inf, -np.inf, 0.0, -0.0, tiny, -tiny, mn, -mn, np.nextafter(mn, 0.0),
                     1.0, np.nextafter(1.0, 2.0), np.nextafter(1.0, 0.0), -1.0,
                     -np.nextafter(1.0, 2.0), -np.nextafter(1.0, 0.0), big, -big, 1e300, -1e300])
    rng = np.random.default_rng(seed)
    n = 200_003
    x = rng.uniform(-1e300, 1e300, n)
    pick = rng.random(n) < 0.3
    x[pick] = pool[rng.integers(0, pool.size, int(pick.sum()))]
    t = torch.from_numpy(x)
    for op in ("min", "max"):
        assert_reduce_matches(run_reduce(mt, t, n, "f64", op), t, n, "f64", op)
        for inclusive in (False, True):
            assert_scan_matches(run_scan(mt, t, n, "f64", op, inclusive), t, n, "f64", op,
                                inclusive=inclusive)
    # Mostly zeros of both signs and the smallest magnitudes: ties everywhere.
    z = pool[rng.integers(2, 6, n)]
    tz = torch.from_numpy(z)
    for op in ("min", "max"):
        assert_reduce_matches(run_reduce(mt, tz, n, "f64", op), tz, n, "f64", op)
        assert_scan_matches(run_scan(mt, tz, n, "f64", op, True), tz, n, "f64", op, inclusive=True)
