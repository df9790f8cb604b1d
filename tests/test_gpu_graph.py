"""Every call only enqueues work on its stream, so a sequence of calls can be
captured once in a CUDA graph and replayed: each replay must compute the
oracle's results for whatever the input buffers hold at that time."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from checks import assert_reduce_matches, assert_rows_close, assert_scan_matches, assert_select_matches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def test_calls_replay_in_a_cuda_graph(mt):
    i32 = torch.int32
    n = 200_003
    short_rows = torch.empty((33, 4099), dtype=torch.bfloat16, device="cuda")
    long_rows = torch.empty((2, 300_001), dtype=torch.float32, device="cuda")
    a = torch.empty(n, dtype=i32, device="cuda")
    v = torch.empty(n, dtype=torch.float32, device="cuda")
    fl = torch.empty(n, dtype=torch.uint8, device="cuda")
    keys = torch.empty(n, dtype=i32, device="cuda")
    vals = torch.empty(n, dtype=i32, device="cuda")
    st = torch.empty((n, 3), dtype=i32, device="cuda")  # 12-byte structs
    sto = torch.empty_like(st)
    num3 = torch.zeros(1, dtype=i32, device="cuda")
    st_scr = mt.alloc_scratch(n, i32, mt.MT_SCRATCH_SELECT)
    so, lo = torch.empty_like(short_rows), torch.empty_like(long_rows)
    ao, vo, ko, kvo = torch.empty_like(a), torch.empty_like(v), torch.empty_like(keys), torch.empty_like(vals)
    red = torch.empty(1, dtype=i32, device="cuda")
    num = torch.zeros(1, dtype=i32, device="cuda")
    nr = torch.zeros(1, dtype=i32, device="cuda")
    nd = torch.tensor([n], dtype=i32, device="cuda")
    scan_scr = mt.alloc_scratch(n, i32, mt.MT_SCRATCH_SCAN)
    red_scr = mt.alloc_scratch(n, i32, mt.MT_SCRATCH_REDUCE)
    sel_scr = mt.alloc_scratch(n, i32, mt.MT_SCRATCH_SELECT)
    rbk_scr = mt.alloc_scratch(n, i32, mt.MT_SCRATCH_REDUCE_BY_KEY)

    def calls():
        mt.mt_scan_rows(short_rows, so, True)
        mt.mt_scan_rows(long_rows, lo, False)  # look-back records from the library's pool
        mt.mt_exclusive_scan(a, ao, scan_scr, nd, "add")
        mt.mt_reduce(a, red, red_scr, nd, "max")
        mt.mt_select(v, fl, vo, num, sel_scr, nd)
        mt.mt_select_wide(st, fl, sto, num3, st_scr, nd)
        mt.mt_reduce_by_key_add(keys, vals, ko, kvo, nr, rbk_scr, nd)

    def fill(seed):
        x = {
            "short": workloads.normal((33, 4099), seed, "bf16"),
            "long": workloads.uniform((2, 300_001), seed + 1, -1.0, 1.0, "f32"),
            "a": workloads.randint((n,), seed + 2, 0, 1000, "i32"),
        }
        x["v"], x["fl"] = workloads.select_inputs(n, 0.3, seed + 3)
        x["keys"], x["vals"] = workloads.runs(n, 5.0, seed + 4, "i32", "i32")
        x["st"] = workloads.randint((n, 3), seed + 5, -(2**31), 2**31 - 1, "i32")
        st.copy_(x["st"])
        short_rows.copy_(x["short"])
        long_rows.copy_(x["long"])
        a.copy_(x["a"])
        v.copy_(x["v"])
        fl.copy_(x["fl"])
        keys.copy_(x["keys"])
        vals.copy_(x["vals"])
        return x

    def check(x):
        assert_rows_close(so, x["short"], "bf16", True)
        assert_rows_close(lo, x["long"], "f32", False)
        assert_scan_matches(ao, x["a"], n, "i32", "add")
        assert_reduce_matches(red, x["a"], n, "i32", "max")
        assert_select_matches(vo, num, x["v"], x["fl"], n)
        ref3, k3 = oracle.select_wide(x["st"].numpy(), x["fl"].numpy(), n, 12)
        assert int(num3.item()) == k3
        assert np.array_equal(sto[:k3].cpu().numpy().view(np.uint8).reshape(k3, 12), ref3)
        want_k, want_v, r = oracle.reduce_by_key_add(x["keys"], x["vals"], n, "i32", "i32")
        assert int(nr.item()) == r
        assert np.array_equal(ko[:r].cpu().numpy(), want_k)
        assert np.array_equal(kvo[:r].cpu().numpy(), want_v)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one eager pass: lazy attributes and pools are set up
        fill(1)
        calls()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    torch.cuda.synchronize()
    for seed in (10, 20):
        x = fill(seed)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert mt.mt_scan_status() == 0
        check(x)
