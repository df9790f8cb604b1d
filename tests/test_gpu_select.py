"""Parity of mt_select (CUDA, through the C ABI) with the CPU oracle."""
import pytest
import torch

import workloads
from checks import assert_select_matches
from golden_io import load_all

pytestmark = pytest.mark.gpu

SENT = 0x7FBADBAD  # a NaN bit pattern: the copy must move bits, not values


@pytest.fixture(scope="module")
def mt():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import prefix_scan_row_gb300 as m
    return m


def run_select(mt, vals_cpu, flags_cpu, n, arr_off=0, flag_off=0, out_off=0):
    cap = vals_cpu.numel()
    abuf = torch.zeros(cap + arr_off, dtype=vals_cpu.dtype, device="cuda")
    arr = abuf[arr_off:]
    arr.copy_(vals_cpu.cuda())
    fbuf = torch.zeros(cap + flag_off, dtype=torch.uint8, device="cuda")
    flags = fbuf[flag_off:]
    flags.copy_(flags_cpu.cuda())
    obuf = torch.full((cap + out_off + 16,), SENT, dtype=torch.int32, device="cuda")
    out = obuf[out_off:out_off + cap].view(vals_cpu.dtype)
    num_out = torch.full((1,), -9, dtype=torch.int32, device="cuda")
    scratch = mt.alloc_scratch(max(cap, 1), torch.int32, mt.MT_SCRATCH_SELECT)
    scratch.fill_(-1)
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    mt.mt_select(arr, flags, out, num_out, scratch, n_dev)
    torch.cuda.synchronize()
    assert mt.mt_scan_status() == 0
    k = int(num_out.item())
    assert torch.all(obuf[out_off + k:] == SENT).item(), "tail of out was touched"
    if out_off:
        assert torch.all(obuf[:out_off] == SENT).item()
    return out, num_out


def test_select_golden(mt):
    g = load_all()["algos_select_i32"]
    vals = torch.tensor(g["arr"], dtype=torch.int32)
    flags = torch.tensor(g["flags"], dtype=torch.uint8)
    out, num = run_select(mt, vals, flags, len(g["arr"]))
    assert int(num.item()) == g["num_out"]
    assert out[:g["num_out"]].cpu().tolist() == g["out"]


@pytest.mark.parametrize("p", [0.0, 0.01, 0.5, 1.0])
@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 255, 8191, 8192, 8193, 100003, (1 << 20) + 3])
def test_select_sizes(mt, p, n):
    cap = n + 29
    vals = workloads.uniform((cap,), n + 3, -1.0, 1.0, "f32")
    flags = workloads.bernoulli_u8(cap, p, n + 4)
    out, num = run_select(mt, vals, flags, n)
    assert_select_matches(out, num, vals, flags, n)


@pytest.mark.parametrize("offs", [(1, 0, 0), (0, 3, 0), (0, 0, 1), (2, 5, 3)])
@pytest.mark.parametrize("p", [0.01, 0.5])
def test_select_misaligned(mt, offs, p):
    n = 60001
    vals = workloads.uniform((n,), 31, -1.0, 1.0, "f32")
    flags = workloads.bernoulli_u8(n, p, 32)
    out, num = run_select(mt, vals, flags, n, *offs)
    assert_select_matches(out, num, vals, flags, n)


@pytest.mark.parametrize("arr_off", [1, 2, 3])
@pytest.mark.parametrize("flag_off", [1, 4, 9, 15])
@pytest.mark.parametrize("n", [1, 8177, 8192, 8193, 2 * 8192 + 15])
@pytest.mark.parametrize("p", [0.5, 1.0])
def test_select_16_byte_phases_at_tile_edges(mt, arr_off, flag_off, n, p):
    """Every tile of a misaligned input takes the masked path; at these sizes
    the flags' copy of a tile also spills into one more 16-byte chunk."""
    vals = workloads.uniform((n,), 33 + n, -1.0, 1.0, "f32")
    flags = workloads.bernoulli_u8(n, p, 34 + n)
    out, num = run_select(mt, vals, flags, n, arr_off, flag_off, arr_off)
    assert_select_matches(out, num, vals, flags, n)


@pytest.mark.parametrize("arr_off", [1, 2, 3])
@pytest.mark.parametrize("n", [16384, 3 * 16384, 3 * 16384 + 5, 100003])
@pytest.mark.parametrize("p", [0.01, 0.3, 0.9, 1.0])
def test_select_aligned_flags_values_off_boundary(mt, arr_off, n, p):
    """Flags at a 16-byte boundary and values 1 to 3 slots past one: the full
    tiles take the chunk-wise packing, which reads each chunk's values from
    the two aligned 16-byte chunks around them; the bit patterns make a
    shift by the wrong number of slots visible."""
    bits = workloads.randint((n,), 51 + arr_off, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(n, p, 52 + n)
    out, num = run_select(mt, bits.view(torch.float32), flags, n, arr_off, 0, 0)
    assert_select_matches(out, num, bits, flags, n)


def test_select_bit_patterns(mt):
    """Any 32-bit pattern (NaNs, -0.0, denormals) is copied unchanged."""
    n = 40000
    bits = workloads.randint((n,), 41, -(2**31), 2**31 - 1, "i32")
    flags = workloads.bernoulli_u8(n, 0.3, 42)
    out, num = run_select(mt, bits.view(torch.float32), flags, n)
    assert_select_matches(out, num, bits, flags, n)


@pytest.mark.parametrize("p", [0.5, 0.01])
def test_select_full_size(mt, p):
    n = workloads.SELECT_N
    vals, flags = workloads.select_inputs(n, p)
    out, num = run_select(mt, vals, flags, n)
    assert_select_matches(out, num, vals, flags, n)
    assert int(num.item()) == int(flags.sum().item())
