"""Host threads that call the library at the same time, each on its own CUDA
stream with its own buffers (the launch path's per-device caches are shared by
all of them): every result must still equal the oracle's."""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads
from checks import assert_reduce_matches, assert_rows_close, assert_scan_matches, assert_select_matches

pytestmark = pytest.mark.gpu

THREADS = 6
REPS = 3


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def make_jobs(mt, t):
    """Thread t's calls as (launch(stream), check()) pairs on buffers of its
    own; sizes differ per thread so that no two calls share a shape."""
    jobs = []
    i32 = torch.int32

    x_cpu = workloads.normal((7 + t, 3001 + 97 * t), 100 + t, "bf16")
    x = x_cpu.cuda()
    xo = torch.empty_like(x)
    jobs.append((lambda s: mt.mt_scan_rows(x, xo, True, stream=s),
                 lambda: assert_rows_close(xo, x_cpu, "bf16", True)))

    cap = 300_007 + 1009 * t
    nd = torch.tensor([cap], dtype=i32, device="cuda")
    a_cpu = workloads.randint((cap,), 200 + t, 0, 16, "i32")
    a = a_cpu.cuda()
    ao = torch.empty_like(a)
    ascr = mt.alloc_scratch(cap, i32, mt.MT_SCRATCH_SCAN)
    jobs.append((lambda s: mt.mt_exclusive_scan(a, ao, ascr, nd, "add", stream=s),
                 lambda: assert_scan_matches(ao, a_cpu, cap, "i32", "add")))

    f_cpu = workloads.uniform((cap,), 300 + t, -1.0, 1.0, "f32")
    f = f_cpu.cuda()
    fr = torch.empty(1, dtype=torch.float32, device="cuda")
    fscr = mt.alloc_scratch(cap, torch.float32, mt.MT_SCRATCH_REDUCE)
    jobs.append((lambda s: mt.mt_reduce(f, fr, fscr, nd, "max", stream=s),
                 lambda: assert_reduce_matches(fr, f_cpu, cap, "f32", "max")))

    v_cpu, fl_cpu = workloads.select_inputs(cap, 0.3, 400 + t)
    v, fl = v_cpu.cuda(), fl_cpu.cuda()
    vo = torch.empty_like(v)
    num = torch.zeros(1, dtype=i32, device="cuda")
    sscr = mt.alloc_scratch(cap, i32, mt.MT_SCRATCH_SELECT)
    jobs.append((lambda s: mt.mt_select(v, fl, vo, num, sscr, nd, stream=s),
                 lambda: assert_select_matches(vo, num, v_cpu, fl_cpu, cap)))

    words = 3 + (t % 3) * 2  # 12-, 20- and 28-byte structs (W = 5, 7 at run time)
    st_cpu = workloads.randint((cap, words), 450 + t, -(2**31), 2**31 - 1, "i32")
    st = st_cpu.cuda()
    sto = torch.empty_like(st)
    num3 = torch.zeros(1, dtype=i32, device="cuda")
    st_scr = mt.alloc_scratch(cap, i32, mt.MT_SCRATCH_SELECT)

    def check_struct():
        ref, k3 = oracle.select_wide(st_cpu.numpy(), fl_cpu.numpy(), cap, 4 * words)
        assert int(num3.item()) == k3
        assert np.array_equal(sto[:k3].cpu().numpy().view(np.uint8).reshape(k3, 4 * words), ref)

    jobs.append((lambda s: mt.mt_select_wide(st, fl, sto, num3, st_scr, nd, stream=s), check_struct))

    k_cpu, kv_cpu = workloads.runs(cap, 6.0, 500 + t, "i32", "i32")
    k, kv = k_cpu.cuda(), kv_cpu.cuda()
    ko, kvo = torch.empty_like(k), torch.empty_like(kv)
    nr = torch.zeros(1, dtype=i32, device="cuda")
    rscr = mt.alloc_scratch(cap, i32, mt.MT_SCRATCH_REDUCE_BY_KEY)

    def check_rbk():
        want_k, want_v, r = oracle.reduce_by_key_add(k_cpu, kv_cpu, cap, "i32", "i32")
        assert int(nr.item()) == r
        assert np.array_equal(ko[:r].cpu().numpy(), want_k)
        assert np.array_equal(kvo[:r].cpu().numpy(), want_v)

    jobs.append((lambda s: mt.mt_reduce_by_key_add(k, kv, ko, kvo, nr, rscr, nd, stream=s), check_rbk))
    return jobs


def test_concurrent_host_threads(mt):
    all_jobs = [make_jobs(mt, t) for t in range(THREADS)]
    torch.cuda.synchronize()  # every buffer is in place before any thread starts
    errors = []
    start = threading.Barrier(THREADS)

    def worker(jobs):
        try:
            s = torch.cuda.Stream()
            start.wait()
            for _ in range(REPS):
                for launch, _ in jobs:
                    launch(s)
            s.synchronize()
        except Exception as e:  # reported after the join
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(jobs,)) for jobs in all_jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    for jobs in all_jobs:
        for _, check in jobs:
            check()
