"""Parity of mt_reduce_by_key_add (CUDA, through the C ABI) with the CPU
oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from checks import ABS, REL
from golden_io import load_all

pytestmark = pytest.mark.gpu

TW = {"i32": torch.int32, "u32": torch.int32, "f32": torch.float32}   # device allocation type
TT = {"i32": torch.int32, "u32": torch.uint32, "f32": torch.float32}  # dtype the call sees
SENT = -123456789


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def to_dev(t, dt, off=0):
    twin = t.view(torch.int32) if t.dtype == torch.uint32 else t
    buf = torch.zeros(t.numel() + off + 4, dtype=twin.dtype, device="cuda")
    buf[off:off + t.numel()].copy_(twin.cuda())
    return buf[off:off + t.numel()].view(TT[dt])


def run(mt, keys, vals, n, kd, vd, off=0):
    cap = keys.numel()
    k = to_dev(keys, kd, off)
    v = to_dev(vals, vd, off)
    kob = torch.full((cap + 8,), SENT, dtype=torch.int32, device="cuda")
    vob = torch.full((cap + 8,), SENT, dtype=torch.int32, device="cuda")
    ko, vo = kob[:cap].view(TT[kd]), vob[:cap].view(TT[vd])
    num = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(max(cap, 1), torch.int32, mt.MT_SCRATCH_REDUCE_BY_KEY)
    scr.fill_(-1)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_reduce_by_key_add(k, v, ko, vo, num, scr, nd)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    r = int(num.item())
    assert torch.all(kob[r:] == SENT).item() and torch.all(vob[r:] == SENT).item(), "tail touched"
    return kob[:r].cpu().numpy(), vob[:r].cpu().numpy(), r


def check(got, keys, vals, n, kd, vd):
    gk, gv, r = got
    ko, vo, rr, s64, m64 = oracle.reduce_by_key_add(keys, vals, n, kd, vd, want_f64=True)
    assert r == rr, f"num_runs {r} != {rr}"
    assert np.array_equal(gk.view(np.uint32), ko.view(np.uint32)), "keys differ"
    if vd == "f32":
        err = np.abs(gv.view(np.float32).astype(np.float64) - s64)
        bad = np.nonzero(~(err <= REL * m64 + ABS))[0]
        assert bad.size == 0, f"{bad.size} run sums out of tolerance; first {bad[0]}"
    else:
        assert np.array_equal(gv.view(np.uint32), vo.view(np.uint32)), "sums differ"


def test_rbk_golden(mt):
    g = load_all()["algos_reduce_by_key_add_i32"]
    keys = torch.tensor(g["keys"], dtype=torch.int32)
    vals = torch.tensor(g["values"], dtype=torch.int32)
    gk, gv, r = run(mt, keys, vals, len(g["keys"]), "i32", "i32")
    assert r == g["num_runs"] and gk.tolist() == g["keys_out"] and gv.tolist() == g["values_out"]


@pytest.mark.parametrize("kd,vd", [("i32", "f32"), ("i32", "i32"), ("u32", "u32"), ("f32", "f32"),
                                   ("f32", "i32")])
@pytest.mark.parametrize("mean_run", [1.0, 3.0, 40.0, 5000.0])
@pytest.mark.parametrize("n", [0, 1, 2, 4095, 4096, 4097, 100003, (1 << 20) + 5])
def test_rbk(mt, kd, vd, mean_run, n):
    keys, vals = workloads.runs(n + 7, mean_run, n + 71, kd, vd)
    check(run(mt, keys, vals, n, kd, vd), keys, vals, n, kd, vd)


@pytest.mark.parametrize("off", [1, 2, 3])
def test_rbk_misaligned(mt, off):
    n = 50001
    keys, vals = workloads.runs(n, 7.0, 73, "i32", "f32")
    check(run(mt, keys, vals, n, "i32", "f32", off=off), keys, vals, n, "i32", "f32")


def test_rbk_float_keys(mt):
    """NaN keys are runs of their own, -0 joins +0, across tile boundaries."""
    n = 20000
    k = np.ones(n, dtype=np.float32)
    k[4090:4100] = np.nan          # ten one-element runs across the first tile edge
    k[8190:8194] = [0.0, -0.0, 0.0, -0.0]
    k[9000:] = 2.0
    keys = torch.from_numpy(k)
    vals = workloads.runs(n, 3.0, 75, "i32", "i32")[1]
    check(run(mt, keys, vals, n, "f32", "i32"), keys, vals, n, "f32", "i32")


def test_rbk_one_long_run_and_all_unique(mt):
    n = 3_000_001
    keys = torch.full((n,), 7, dtype=torch.int32)
    vals = workloads.randint((n,), 77, 1 << 28, 1 << 30, "i32")  # the sum wraps
    check(run(mt, keys, vals, n, "i32", "i32"), keys, vals, n, "i32", "i32")
    keys = torch.arange(n, dtype=torch.int32)
    check(run(mt, keys, vals, n, "i32", "i32"), keys, vals, n, "i32", "i32")


def test_rbk_full_size(mt):
    n = 1 << 26
    keys, vals = workloads.runs(n, 8.0, 79, "i32", "f32")
    check(run(mt, keys, vals, n, "i32", "f32"), keys, vals, n, "i32", "f32")
