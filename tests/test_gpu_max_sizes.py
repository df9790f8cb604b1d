"""Maximum sizes: a row scan of more than 2^31 elements (64-bit row offsets),
and the 1-D calls at the largest live count an int32 n_dev can hold. The
inputs are drawn on the device from seeded generators; the results are
checked on the device by properties that fix them exactly, and sampled rows
against the oracle."""
import pytest
import torch

from checks import assert_rows_close

pytestmark = pytest.mark.gpu

N_MAX = 2**31 - 1  # the largest int32 live count


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def gen(seed):
    return torch.Generator(device="cuda").manual_seed(seed)


def test_rows_past_2p31_elements(mt):
    rows, n = 32768, 65539  # 2.15e9 bf16 elements; ragged, misaligned rows
    x = torch.randn((rows, n), device="cuda", generator=gen(1)).to(torch.bfloat16)
    out = torch.empty_like(x)
    mt.mt_scan_rows(x, out, False)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    for r in (0, 1, 12345, rows - 1):
        assert_rows_close(out[r:r + 1].cpu(), x[r:r + 1].cpu(), "bf16", False)
    del x, out
    torch.cuda.empty_cache()


def test_exclusive_scan_at_int32_limit(mt):
    x = torch.randint(0, 16, (N_MAX,), device="cuda", generator=gen(2), dtype=torch.int32)
    out = torch.empty_like(x)
    scr = mt.alloc_scratch(N_MAX, torch.int32, mt.MT_SCRATCH_SCAN)
    nd = torch.tensor([N_MAX], dtype=torch.int32, device="cuda")
    mt.mt_exclusive_scan(x, out, scr, nd, "add")
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    # out[0] = 0 and out[i+1] - out[i] = x[i] (wrapping) fix every output
    assert out[0].item() == 0
    assert torch.equal(out[1:] - out[:-1], x[:-1])
    del x, out, scr
    torch.cuda.empty_cache()


def test_select_at_int32_limit(mt):
    v = torch.randint(-(2**31), 2**31 - 1, (N_MAX,), device="cuda", generator=gen(3), dtype=torch.int32)
    f = (torch.rand((N_MAX,), device="cuda", generator=gen(4)) < 0.5).to(torch.uint8)
    out = torch.empty_like(v)
    num = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(N_MAX, torch.int32, mt.MT_SCRATCH_SELECT)
    nd = torch.tensor([N_MAX], dtype=torch.int32, device="cuda")
    mt.mt_select(v, f, out, num, scr, nd)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    want = v[f.bool()]
    k = int(num.item())
    assert k == want.numel()
    assert torch.equal(out[:k], want)
    del v, f, out, want, scr
    torch.cuda.empty_cache()


def test_reduce_by_key_at_int32_limit(mt):
    n = N_MAX
    starts = torch.rand((n,), device="cuda", generator=gen(5)) < 0.125
    starts[0] = True
    keys = (torch.cumsum(starts.to(torch.int64), 0) % 7).to(torch.int32)  # neighbouring runs differ
    vals = torch.randint(-1000, 1000, (n,), device="cuda", generator=gen(6), dtype=torch.int32)
    ko, vo = torch.empty_like(keys), torch.empty_like(vals)
    nr = torch.zeros(1, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_REDUCE_BY_KEY)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_reduce_by_key_add(keys, vals, ko, vo, nr, scr, nd)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    head = torch.nonzero(starts).flatten()  # run starts (keys change exactly there)
    r = head.numel()
    assert int(nr.item()) == r
    assert torch.equal(ko[:r], keys[head])
    cs = torch.cumsum(vals.to(torch.int64), 0)
    ends = torch.cat([head[1:] - 1, torch.tensor([n - 1], device="cuda")])
    before = torch.where(head > 0, cs[(head - 1).clamp(min=0)], torch.zeros_like(head))
    sums = ((cs[ends] - before) & 0xFFFFFFFF).to(torch.int64)
    sums = torch.where(sums >= 2**31, sums - 2**32, sums).to(torch.int32)
    assert torch.equal(vo[:r], sums)
    del keys, vals, ko, vo, scr, cs
    torch.cuda.empty_cache()
