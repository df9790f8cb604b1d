"""The bounds-checked build (libmtscan_checked.so) on small, ragged, misaligned
and timeout-path cases.

That build's kernels check every global store and every shared-memory access
against the buffer it belongs to; an access outside it is skipped and
recorded as MT_ERR_BOUNDS, which mt_scan_status() reports. It stands in for a
memory checker: every case here must give the oracle's result with the
status word clear (or, on the timeout path, the timeout and then a correct
call). The cases are those where index arithmetic goes wrong first: sizes
around tile boundaries, row starts and arrays off their 16-byte boundaries,
live counts below the capacity, and the prefixes that a look-back which gave
up leaves incomplete.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from checks import (assert_reduce_matches, assert_rows_close, assert_rows_op_close, assert_scan_matches,
                    assert_select_matches)

pytestmark = pytest.mark.gpu


class _Checked:
    """The checked library's calls, with the package's constants."""

    def __init__(self, mod, lib):
        self._mod, self._lib = mod, lib

    def __getattr__(self, name):
        return getattr(self._lib, name) if hasattr(self._lib, name) else getattr(self._mod, name)


@pytest.fixture(scope="module")
def ck():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    lib = m.load_checked()
    assert lib.mt_scan_build_checked(), "the checked library was not built with its checks"
    assert lib.mt_scan_status() == 0
    return _Checked(m, lib)


def _on_device(x_cpu, off):
    """x_cpu copied to the device `off` elements past a 16-byte boundary."""
    flat = x_cpu.reshape(-1)
    buf = torch.zeros(flat.numel() + off + 16, dtype=flat.dtype, device="cuda")
    v = buf[off:off + flat.numel()]
    v.copy_(flat.cuda())
    return v.view(x_cpu.shape)


def _rows_input(dtype, shape, seed):
    if dtype == "f32":
        return workloads.uniform(shape, seed, -1.0, 1.0, "f32")
    return workloads.normal(shape, seed, dtype)


ROW_SHAPES = [(1, 1), (3, 5), (4, 4099), (2, 16384), (2, 16385), (2, 100003), (1, (1 << 20) + 3)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", ROW_SHAPES)
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("off", [0, 1])
def test_checked_rows(ck, dtype, shape, inclusive, off):
    x_cpu = _rows_input(dtype, shape, 3 + shape[1])
    x = _on_device(x_cpu, off)
    out = torch.empty_like(x)
    ck.mt_scan_rows(x, out, inclusive)
    assert ck.mt_scan_status() == 0
    assert_rows_close(out, x_cpu, dtype, inclusive)


@pytest.mark.parametrize("op", ["mul", "max", "min"])
@pytest.mark.parametrize("dtype,shape", [("bf16", (5, 4099)), ("f32", (2, 100003))])
def test_checked_rows_op(ck, op, dtype, shape):
    x_cpu = workloads.near_one(shape, 21, dtype) if op == "mul" else _rows_input(dtype, shape, 22)
    x = x_cpu.cuda()
    out = torch.empty_like(x)
    ck.mt_scan_rows_op(x, out, op, True)
    assert ck.mt_scan_status() == 0
    assert_rows_op_close(out, x_cpu, dtype, op, True)


TWIN = {"i32": torch.int32, "i64": torch.int64, "f32": torch.float32, "u32": torch.int32,
        "u64": torch.int64, "f64": torch.float64}
TDT = {"i32": torch.int32, "i64": torch.int64, "f32": torch.float32, "u32": torch.uint32,
       "u64": torch.uint64, "f64": torch.float64}


def _scan_input(dtype, cap, seed):
    if dtype in ("u32", "u64"):
        return workloads.bits_uniform((cap,), seed, dtype)
    if dtype == "f64":
        return workloads.uniform64((cap,), seed, -1.0, 1.0)
    if dtype == "f32":
        return workloads.uniform((cap,), seed, -1.0, 1.0, "f32")
    return workloads.randint((cap,), seed, -1000, 1000, dtype)


def _dev_1d(dtype, x_cpu, off):
    twin = x_cpu.view(TWIN[dtype]) if dtype in ("u32", "u64") else x_cpu
    return _on_device(twin, off).view(TDT[dtype])


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32", "u32", "u64", "f64"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("n,off", [(0, 0), (1, 1), (37, 0), (12289, 1), (100003, 3)])
def test_checked_scan_and_reduce(ck, dtype, op, n, off):
    cap = n + 5  # live count below the capacity
    x_cpu = _scan_input(dtype, cap, 40 + n)
    arr = _dev_1d(dtype, x_cpu, off)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    scr = ck.alloc_scratch(cap, TDT[dtype], ck.MT_SCRATCH_SCAN)
    scr.fill_(-1)
    for inclusive in (False, True):
        out = torch.zeros(cap, dtype=TWIN[dtype], device="cuda").view(TDT[dtype])
        (ck.mt_inclusive_scan if inclusive else ck.mt_exclusive_scan)(arr, out, scr, n_dev, op)
        assert ck.mt_scan_status() == 0
        assert_scan_matches(out, x_cpu, n, dtype, op, inclusive=inclusive)
    r = torch.zeros(1, dtype=TWIN[dtype], device="cuda").view(TDT[dtype])
    rscr = ck.alloc_scratch(cap, TDT[dtype], ck.MT_SCRATCH_REDUCE)
    ck.mt_reduce(arr, r, rscr, n_dev, op)
    assert ck.mt_scan_status() == 0
    assert_reduce_matches(r, x_cpu, n, dtype, op)


@pytest.mark.parametrize("n", [1, 8191, 8193, 16385, 100003])
@pytest.mark.parametrize("p", [0.5, 0.01])
@pytest.mark.parametrize("voff,foff", [(0, 0), (1, 0), (2, 0), (3, 0), (0, 3), (3, 5)])
def test_checked_select(ck, n, p, voff, foff):
    vals, flags = workloads.select_inputs(n, p, seed=50 + n)
    v = _on_device(vals, voff)
    f = _on_device(flags, foff)
    out = torch.zeros(n + 8, dtype=torch.float32, device="cuda")
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = ck.alloc_scratch(n, torch.int32, ck.MT_SCRATCH_SELECT)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    ck.mt_select(v, f, out, num, scr, nd)
    assert ck.mt_scan_status() == 0
    assert_select_matches(out, num, vals, flags, n)


@pytest.mark.parametrize("words", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("n,p", [(1, 0.5), (8193, 0.5), (100003, 0.01)])
def test_checked_select_wide(ck, words, n, p):
    vals = workloads.randint((n, words), 60 + words, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(n, p, 61)
    if words == 2:  # 8-byte elements
        vals = vals.view(torch.int64).reshape(n)
    v, f = vals.cuda(), flags.cuda()
    out = torch.zeros_like(v)
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = ck.alloc_scratch(n, torch.int32, ck.MT_SCRATCH_SELECT)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    ck.mt_select_wide(v, f, out, num, scr, nd)
    assert ck.mt_scan_status() == 0
    want = vals[flags.bool()]
    assert int(num.item()) == want.shape[0]
    assert torch.equal(out[:want.shape[0]].cpu(), want)


@pytest.mark.parametrize("kd,vd", [("i32", "i32"), ("f32", "f32"), ("i32", "f32")])
@pytest.mark.parametrize("n,off", [(1, 0), (6145, 0), (100003, 1)])
def test_checked_reduce_by_key(ck, kd, vd, n, off):
    keys, vals = workloads.runs(n, 6.0, 70 + n, kd, vd)
    k = _on_device(keys, off)
    v = _on_device(vals, off)  # keys and values share their 16-byte phase
    ko, vo = torch.zeros_like(k), torch.zeros_like(v)
    nr = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = ck.alloc_scratch(n, torch.int32, ck.MT_SCRATCH_REDUCE_BY_KEY)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    ck.mt_reduce_by_key_add(k, v, ko, vo, nr, scr, nd)
    assert ck.mt_scan_status() == 0
    want_k, want_v, r = oracle.reduce_by_key_add(keys, vals, n, kd, vd)
    assert int(nr.item()) == r
    assert np.array_equal(ko[:r].cpu().view(torch.int32).numpy().view(np.uint32), want_k.view(np.uint32))
    if vd == "f32":
        mag = np.abs(vals.numpy().astype(np.float64))
        got = vo[:r].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - want_v.astype(np.float64)) <= 1e-5 * mag.sum() + 1e-6)
    else:
        assert np.array_equal(vo[:r].cpu().numpy(), want_v)


@pytest.mark.parametrize("dtype,shape", [("f32", (2, 100003)), ("bf16", (3, 70001))])
def test_checked_rows_noalloc(ck, dtype, shape):
    x_cpu = _rows_input(dtype, shape, 80)
    x = x_cpu.cuda()
    out = torch.empty_like(x)
    ck.mt_scan_rows_noalloc(x, out, True)
    assert ck.mt_scan_status() == 0
    assert_rows_close(out, x_cpu, dtype, True)


# The timeout path: one tile never publishes, its successors give up with
# incomplete prefixes and carry on; every access must still stay in bounds
# (the error word then holds the timeout, recorded first), and the next call
# must be correct again.
def _timeout_then(ck, call, tile=2):
    try:
        ck.mt_scan_debug_lookback(skip_publish_tile=tile, spin_limit=4096)
        call()
        assert ck.mt_scan_status() == ck.MT_ERR_LOOKBACK_TIMEOUT
    finally:
        ck.mt_scan_debug_lookback(-1, 0)
    assert ck.mt_scan_status() == 0
    call()
    assert ck.mt_scan_status() == 0


@pytest.mark.parametrize("dtype", ["i32", "i64", "f64"])
def test_checked_scan_timeout(ck, dtype):
    n = 1 << 20
    x_cpu = _scan_input(dtype, n, 90)
    arr = x_cpu.cuda()
    out = torch.zeros_like(arr)
    scr = ck.alloc_scratch(n, arr.dtype, ck.MT_SCRATCH_SCAN)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    _timeout_then(ck, lambda: ck.mt_exclusive_scan(arr, out, scr, nd, "add"))
    assert_scan_matches(out, x_cpu, n, dtype, "add")


def test_checked_rows_timeout(ck):
    x_cpu = workloads.rows_long(rows=2, n=1 << 18)
    x = x_cpu.cuda()
    out = torch.empty_like(x)
    _timeout_then(ck, lambda: ck.mt_scan_rows(x, out, True))
    assert_rows_close(out, x_cpu, "f32", True)


@pytest.mark.parametrize("kind", ["f32", "f64", "struct3"])
def test_checked_select_timeout(ck, kind):
    n = 1 << 20
    vals, flags = workloads.select_inputs(n, 0.5, seed=91)
    if kind == "f64":
        vals = vals.to(torch.float64)
    elif kind == "struct3":
        vals = workloads.randint((n, 3), 92, -(2**31), 2**31 - 1, "i32")
    v, f = vals.cuda(), flags.cuda()
    out = torch.zeros_like(v)
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = ck.alloc_scratch(n, torch.int32, ck.MT_SCRATCH_SELECT)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    _timeout_then(ck, lambda: ck.mt_select_wide(v, f, out, num, scr, nd))
    want = vals[flags.bool()]
    assert int(num.item()) == want.shape[0]
    assert torch.equal(out[:want.shape[0]].cpu(), want)


def test_checked_reduce_by_key_timeout(ck):
    """The path on which an incomplete prefix once produced the run index
    2^32 - 1: every output index must stay in bounds."""
    n = 1 << 20
    keys, vals = workloads.runs(n, 8.0, 93, "i32", "i32")
    k, v = keys.cuda(), vals.cuda()
    ko, vo = torch.zeros_like(k), torch.zeros_like(v)
    nr = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = ck.alloc_scratch(n, torch.int32, ck.MT_SCRATCH_REDUCE_BY_KEY)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    _timeout_then(ck, lambda: ck.mt_reduce_by_key_add(k, v, ko, vo, nr, scr, nd), tile=4)
    want_k, want_v, r = oracle.reduce_by_key_add(keys, vals, n, "i32", "i32")
    assert int(nr.item()) == r
    assert np.array_equal(ko[:r].cpu().numpy(), want_k) and np.array_equal(vo[:r].cpu().numpy(), want_v)
