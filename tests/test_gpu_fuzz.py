"""Seeded random cases for every call: random sizes (log-uniform, so tiny,
ragged, tile-boundary and multi-tile cases all occur), dtypes, operations,
inclusive/exclusive forms and misaligned buffer offsets, each compared with
the oracle. The fixed shape lists of the other tests pin known edges; these
cases reach the planners' and the kernels' other paths."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from checks import assert_reduce_matches, assert_rows_op_close, assert_scan_matches, assert_select_matches

pytestmark = pytest.mark.gpu

TWIN = {torch.uint32: torch.int32, torch.uint64: torch.int64}
DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "i32": torch.int32,
      "i64": torch.int64, "u32": torch.uint32, "u64": torch.uint64, "f64": torch.float64}


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def log_uniform(rng, lo, hi):
    return int(round(np.exp(rng.uniform(np.log(lo), np.log(hi)))))


def to_dev(x_cpu, off, fill=0):
    """A device copy of x_cpu starting `off` elements into a larger buffer
    (unsigned tensors go through their signed twins)."""
    twin = TWIN.get(x_cpu.dtype, x_cpu.dtype)
    buf = torch.full((x_cpu.numel() + off + 16,), fill, dtype=twin, device="cuda")
    buf[off:off + x_cpu.numel()].copy_(x_cpu.reshape(-1).view(twin).cuda())
    return buf[off:off + x_cpu.numel()].view(x_cpu.dtype).view(x_cpu.shape)


def input_1d(dtype, cap, seed):
    if dtype in ("u32", "u64"):
        return workloads.bits_uniform((cap,), seed, dtype)
    if dtype == "f64":
        return workloads.uniform64((cap,), seed, -1.0, 1.0)
    lo, hi = {"i32": (-1000, 1000), "i64": (-(1 << 40), 1 << 40)}.get(dtype, (None, None))
    if lo is not None:
        return workloads.randint((cap,), seed, lo, hi, dtype)
    return workloads.uniform((cap,), seed, -1.0, 1.0, "f32")


@pytest.mark.parametrize("case", range(40))
def test_fuzz_rows(mt, case):
    rng = np.random.default_rng(1000 + case)
    dtype = ["f32", "bf16", "f16"][rng.integers(3)]
    op = ["add", "add", "mul", "max", "min"][rng.integers(5)]
    inclusive = bool(rng.integers(2))
    rows = int(rng.integers(1, 8))
    n = log_uniform(rng, 1, 70000)
    if op == "mul":
        x_cpu = workloads.near_one((rows, n), 2000 + case, dtype)
    else:
        x_cpu = workloads.normal((rows, n), 2000 + case, dtype)
    x = to_dev(x_cpu, int(rng.integers(8)))
    out = to_dev(torch.zeros_like(x_cpu), int(rng.integers(8)))
    mt.mt_scan_rows_op(x, out, op, inclusive)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    assert_rows_op_close(out, x_cpu, dtype, op, inclusive)


@pytest.mark.parametrize("case", range(40))
def test_fuzz_scan_and_reduce(mt, case):
    rng = np.random.default_rng(3000 + case)
    dtype = ["i32", "i64", "f32", "u32", "u64", "f64"][rng.integers(6)]
    op = ["add", "min", "max"][rng.integers(3)]
    inclusive = bool(rng.integers(2))
    cap = log_uniform(rng, 1, 1 << 21)
    n = int(rng.integers(0, cap + 1))
    a_cpu = input_1d(dtype, cap, 4000 + case)
    arr = to_dev(a_cpu, int(rng.integers(4)))
    out = to_dev(torch.zeros_like(a_cpu), int(rng.integers(4)))
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(cap, DT[dtype], mt.MT_SCRATCH_SCAN)
    scr.fill_(-1)
    (mt.mt_inclusive_scan if inclusive else mt.mt_exclusive_scan)(arr, out, scr, nd, op)
    red = to_dev(torch.zeros(1, dtype=DT[dtype]), 0)
    rscr = mt.alloc_scratch(cap, DT[dtype], mt.MT_SCRATCH_REDUCE)
    mt.mt_reduce(arr, red, rscr, nd, op)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    assert_scan_matches(out, a_cpu, n, dtype, op, inclusive=inclusive)
    if n > 0:
        assert_reduce_matches(red, a_cpu, n, dtype, op)


@pytest.mark.parametrize("case", range(16))
def test_fuzz_select(mt, case):
    rng = np.random.default_rng(5000 + case)
    n = log_uniform(rng, 1, 1 << 21)
    p = [0.0, 0.01, 0.3, 0.9, 1.0][rng.integers(5)]
    wide = bool(rng.integers(2))
    v_cpu, f_cpu = workloads.select_inputs(n, p, 6000 + case)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    num = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
    if wide:  # 8-byte elements at any 8-byte offsets
        v64 = v_cpu.to(torch.float64)
        arr, fl = to_dev(v64, int(rng.integers(2))), to_dev(f_cpu, int(rng.integers(16)))
        out = to_dev(torch.zeros_like(v64), int(rng.integers(2)))
        mt.mt_select_wide(arr, fl, out, num, scr, nd)
        torch.cuda.synchronize()
        assert mt.mt_scan_status() == 0
        want = v64[f_cpu.bool()]
        k = int(num.item())
        assert k == want.numel()
        assert torch.equal(out[:k].cpu().view(torch.int64), want.view(torch.int64))
    else:  # 4-byte elements at any offsets
        arr = to_dev(v_cpu, int(rng.integers(4)))
        fl = to_dev(f_cpu, int(rng.integers(16)))
        out = to_dev(torch.zeros_like(v_cpu), int(rng.integers(4)))
        mt.mt_select(arr, fl, out, num, scr, nd)
        torch.cuda.synchronize()
        assert mt.mt_scan_status() == 0
        assert_select_matches(out, num, v_cpu, f_cpu, n)


@pytest.mark.parametrize("case", range(16))
def test_fuzz_select_struct(mt, case):
    """Struct elements of 3 to 64 words at random 4-byte offsets of arr and
    out, flags at any offset, every selection density from none to all."""
    rng = np.random.default_rng(6500 + case)
    words = [3, 4, 5, 6, 7, 8, 12, 33, 64][rng.integers(9)]
    n = log_uniform(rng, 1, (1 << 22) // words)
    p = [0.0, 0.003, 0.05, 0.3, 0.9, 1.0][rng.integers(6)]
    vals = workloads.randint((n * words,), 6600 + case, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(n, p, 6700 + case)
    arr = to_dev(vals, int(rng.integers(4))).view(n, words)
    fl = to_dev(flags, int(rng.integers(16)))
    out = to_dev(torch.zeros_like(vals), int(rng.integers(4))).view(n, words)
    num = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_select_wide(arr, fl, out, num, scr, nd)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    ref, k = oracle.select_wide(vals.numpy(), flags.numpy(), n, 4 * words)
    assert int(num.item()) == k
    got = out[:k].cpu().numpy().view(np.uint8).reshape(k, 4 * words)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("case", range(16))
def test_fuzz_reduce_by_key(mt, case):
    rng = np.random.default_rng(7000 + case)
    n = log_uniform(rng, 1, 1 << 21)
    mean_run = [1.0, 2.5, 8.0, 100.0, 1e5][rng.integers(5)]
    kd, vd = [("i32", "i32"), ("i32", "f32"), ("u32", "u32"), ("f32", "i32")][rng.integers(4)]
    keys, vals = workloads.runs(n, mean_run, 8000 + case, kd, vd)
    off = int(rng.integers(4))  # keys and values share their 16-byte phase
    k, v = to_dev(keys, off), to_dev(vals, off)
    ko, vo = to_dev(torch.zeros_like(keys), 0), to_dev(torch.zeros_like(vals), 0)
    nr = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_REDUCE_BY_KEY)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_reduce_by_key_add(k, v, ko, vo, nr, scr, nd)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    want_k, want_v, r, s64, m64 = oracle.reduce_by_key_add(keys, vals, n, kd, vd, want_f64=True)
    assert int(nr.item()) == r
    got_k = ko[:r].cpu().reshape(-1).view(TWIN.get(keys.dtype, keys.dtype)).numpy()
    assert np.array_equal(got_k.view(np.uint32), want_k.view(np.uint32))
    got_v = vo[:r].cpu().reshape(-1).view(TWIN.get(vals.dtype, vals.dtype)).numpy()
    if vd == "f32":
        err = np.abs(got_v.astype(np.float64) - s64)
        assert np.all(err <= 1e-5 * m64 + 1e-6)
    else:
        assert np.array_equal(got_v.view(np.uint32), want_v.view(np.uint32))
