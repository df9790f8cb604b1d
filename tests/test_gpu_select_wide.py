"""Parity of mt_select_wide (8-byte elements; CUDA, through the C ABI) with
the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from golden_io import load_all

pytestmark = pytest.mark.gpu

SENT = -0x0BADBAD0BADBAD0  # sentinel 64-bit pattern


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def run_select64(mt, vals_cpu, flags_cpu, n, out_off=0):
    cap = vals_cpu.numel()
    arr = vals_cpu.cuda()
    flags = flags_cpu.cuda()
    obuf = torch.full((cap + out_off + 16,), SENT, dtype=torch.int64, device="cuda")
    out = obuf[out_off:out_off + cap].view(vals_cpu.dtype)
    num_out = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    scratch = mt.alloc_scratch(max(cap, 1), torch.int32, mt.MT_SCRATCH_SELECT)
    scratch.fill_(-1)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_select_wide(arr, flags, out, num_out, scratch, n_dev)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    k = int(num_out.item())
    assert torch.all(obuf[out_off + k:] == SENT).item(), "tail of out was touched"
    if out_off:
        assert torch.all(obuf[:out_off] == SENT).item()
    return out, k


def check(out, k, vals_cpu, flags_cpu, n):
    ref, kr = oracle.select_wide(vals_cpu, flags_cpu, n, 8)
    assert k == kr, f"num_out {k} != {kr}"
    got = out[:k].detach().cpu().contiguous().view(torch.int64).numpy().view(np.uint64)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches; first at {bad[0]}"


def test_select_wide_golden(mt):
    g = load_all()["algos_select_i32"]
    vals = torch.tensor(g["arr"], dtype=torch.int64)
    flags = torch.tensor(g["flags"], dtype=torch.uint8)
    out, k = run_select64(mt, vals, flags, len(g["arr"]))
    assert k == g["num_out"] and out[:k].cpu().tolist() == g["out"]


@pytest.mark.parametrize("p", [0.0, 0.01, 0.5, 1.0])
@pytest.mark.parametrize("n", [0, 1, 17, 8191, 8192, 8193, 100003, (1 << 20) + 3])
def test_select_wide_sizes(mt, p, n):
    cap = n + 29
    vals = workloads.randint((cap,), n + 5, -(2**62), 2**62, "i64")
    flags = workloads.bernoulli_u8(cap, p, n + 6)
    out, k = run_select64(mt, vals, flags, n)
    check(out, k, vals, flags, n)


def test_select_wide_f64_bits_and_out_offset(mt):
    """f64 elements move as bits (NaN payloads and -0 included); out may be
    8-byte aligned only."""
    n = 300001
    bits = workloads.randint((n,), 61, -(2**62), 2**62, "i64")
    bits[::7] = 0x7FF8DEADBEEF0001  # NaN payloads
    bits[::11] = -(2**63)           # -0.0
    vals = bits.view(torch.float64)
    flags = workloads.bernoulli_u8(n, 0.4, 62)
    out, k = run_select64(mt, vals, flags, n, out_off=1)
    check(out, k, vals, flags, n)


def test_select_wide_full_size(mt):
    """2^26 8-byte elements at p = 0.5."""
    n = 1 << 26
    vals = workloads.randint((n,), 63, -(2**62), 2**62, "i64")
    flags = workloads.bernoulli_u8(n, 0.5, 64)
    out, k = run_select64(mt, vals, flags, n)
    check(out, k, vals, flags, n)


@pytest.mark.parametrize("arr_off", [0, 1])
@pytest.mark.parametrize("flag_off", [0, 1, 8, 15])
@pytest.mark.parametrize("n", [1, 8177, 8192, 8193, 3 * 8192 - 1])
def test_select_wide_any_16_byte_phase(mt, arr_off, flag_off, n):
    """Values 8 bytes past a 16-byte boundary and flags at any offset: the
    bulk copies start at the boundary below and the tile's ends are masked
    (n covers the tile size and the sizes where the flags' copy of a tile
    spills into one more 16-byte chunk)."""
    vals = workloads.randint((n,), 70 + n, -(2**62), 2**62, "i64")
    for p in (0.5, 1.0):
        flags = workloads.bernoulli_u8(n, p, 71 + n)
        abuf = torch.zeros(n + arr_off, dtype=torch.int64, device="cuda")
        arr = abuf[arr_off:]
        arr.copy_(vals.cuda())
        fbuf = torch.zeros(n + flag_off, dtype=torch.uint8, device="cuda")
        fl = fbuf[flag_off:]
        fl.copy_(flags.cuda())
        obuf = torch.full((n + 17,), SENT, dtype=torch.int64, device="cuda")
        out = obuf[1:n + 1]
        num = torch.full((1,), -9, dtype=torch.int32, device="cuda")
        scr = mt.alloc_scratch(n, torch.int32, mt.MT_SCRATCH_SELECT)
        nd = torch.tensor([n], dtype=torch.int32, device="cuda")
        mt.mt_select_wide(arr, fl, out, num, scr, nd)
        torch.cuda.synchronize()
        assert mt.mt_scan_status() == 0
        k = int(num.item())
        assert obuf[0].item() == SENT and torch.all(obuf[1 + k:] == SENT).item()
        check(out, k, vals, flags, n)


def run_select_struct(mt, vals, flags, n, arr_off=0, flag_off=0, out_off=0):
    """vals: [cap, W] int32 on the CPU (one struct per row); the device
    copies start arr_off / flag_off / out_off elements (32-bit words for
    arr and out, bytes for flags) past a 16-byte boundary."""
    cap, words = vals.shape
    abuf = torch.zeros(cap * words + arr_off, dtype=torch.int32, device="cuda")
    arr = abuf[arr_off:].view(cap, words)
    arr.copy_(vals.cuda())
    fbuf = torch.zeros(cap + flag_off, dtype=torch.uint8, device="cuda")
    fl = fbuf[flag_off:]
    fl.copy_(flags.cuda())
    obuf = torch.full((cap * words + out_off + 16,), 0x7BADBAD0, dtype=torch.int32, device="cuda")
    out = obuf[out_off:out_off + cap * words].view(cap, words)
    num = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    scr = mt.alloc_scratch(max(cap, 1), torch.int32, mt.MT_SCRATCH_SELECT)
    scr.fill_(-1)
    nd = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_select_wide(arr, fl, out, num, scr, nd)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    k = int(num.item())
    assert torch.all(obuf[out_off + k * words:] == 0x7BADBAD0).item(), "tail of out was touched"
    assert torch.all(obuf[:out_off] == 0x7BADBAD0).item()
    ref, kr = oracle.select_wide(vals.numpy(), flags.numpy(), n, 4 * words)
    assert k == kr, f"num_out {k} != {kr}"
    got = out[:k].cpu().contiguous().numpy().view(np.uint8).reshape(k, 4 * words)
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} mismatched structs; first at {bad[0] if bad.size else -1}"


@pytest.mark.parametrize("words", [3, 4, 5, 6, 8, 64])  # 12 to 256 bytes; 5 and 64: W at run time
@pytest.mark.parametrize("n", [0, 1, 17, 8191, 8192, 8193, 100003])
@pytest.mark.parametrize("p", [0.01, 0.5, 1.0])
def test_select_struct_sizes(mt, words, n, p):
    cap = n + 29
    if words == 64 and n > 10000:
        cap = n + 1
    vals = workloads.randint((cap, words), n + 7 * words, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(cap, p, n + 8)
    run_select_struct(mt, vals, flags, n)


@pytest.mark.parametrize("words", [3, 4, 5, 8])
@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 7, 0), (0, 0, 3), (3, 15, 1)])
@pytest.mark.parametrize("n", [8177, 8193, 3 * 8192 - 1])
def test_select_struct_offsets_and_tile_edges(mt, words, offs, n):
    """arr and out 4 bytes to 12 bytes past a 16-byte boundary, flags at any
    offset; the sizes put the flags' extra 16-byte chunk at a tile's end."""
    vals = workloads.randint((n, words), 90 + words, -(2**31), 2**31 - 1, "i32")
    for p in (0.5, 1.0):
        flags = workloads.bernoulli_u8(n, p, 91 + n)
        run_select_struct(mt, vals, flags, n, *offs)


def test_select_struct_large(mt):
    """2^24 12-byte structs (a 3-word vector) at p = 0.5; successive
    structs start at every 4-byte phase of a 16-byte boundary."""
    n = 1 << 24
    vals = workloads.randint((n, 3), 95, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(n, 0.5, 96)
    run_select_struct(mt, vals, flags, n)


def test_select_struct_float_fields_move_as_bits(mt):
    """A 16-byte struct of f32 fields (NaN payloads, -0.0) copied bit for bit."""
    n = 50000
    bits = workloads.randint((n, 4), 97, -(2**31), 2**31 - 1, "i32")
    bits[::5, 1] = 0x7FC0BEEF
    bits[::3, 2] = -(2**31)
    flags = workloads.bernoulli_u8(n, 0.3, 98)
    run_select_struct(mt, bits, flags, n)
