"""The all-core CPU scans that bench.py reports as a second CPU baseline must
compute the scans: the row scan checked against the oracle with the GPU
path's tolerances and its bf16/f16 rounding against torch's conversions, the
1-D exclusive scan against the oracle (bit-exact for integers and min/max,
the f32 add bound otherwise)."""
import numpy as np
import pytest
import torch

import workloads
from checks import assert_rows_close
import oracle
from baselines import allcore


def as_tensor(y, dtype):
    if dtype == "f32":
        return torch.from_numpy(y)
    return torch.from_numpy(y.view(np.int16)).view(torch.bfloat16 if dtype == "bf16" else torch.float16)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("inclusive", [True, False])
@pytest.mark.parametrize("shape,threads", [((7, 4099), 3), ((1, 1), 8), ((5, 33), 1), ((64, 1000), 16)])
def test_allcore_matches_oracle(dtype, inclusive, shape, threads):
    x = workloads.normal(shape, 40 + shape[1], dtype)
    y = allcore.scan_rows(x, dtype, inclusive, threads)
    assert_rows_close(as_tensor(y, dtype), x, dtype, inclusive)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_allcore_rounding_is_torchs(dtype):
    """Two-element inclusive rows: out[1] = RN(x0 + x1) with the sum in f32,
    over values spanning subnormals to overflow."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    g = torch.Generator().manual_seed(7)
    bits = torch.randint(-(2 ** 15), 2 ** 15, (200000, 2), generator=g, dtype=torch.int16)
    x = bits.view(tdt)
    finite = torch.isfinite(x.float()).all(dim=1)
    x = x[finite].contiguous()
    y = as_tensor(allcore.scan_rows(x, dtype, True, 4), dtype)
    want = (x[:, 0].float() + x[:, 1].float()).to(tdt)
    got, ref = y[:, 1].view(torch.int16), want.view(torch.int16)
    nan = torch.isnan(want.float())
    assert torch.equal(got[~nan], ref[~nan])
    # out[0] = RN(0 + x0): the value itself, except that -0 becomes +0
    assert torch.equal(y[:, 0].view(torch.int16), (0.0 + x[:, 0].float()).to(tdt).view(torch.int16))


@pytest.mark.parametrize("dtype", ["i32", "i64", "f32"])
@pytest.mark.parametrize("op", ["add", "min", "max"])
@pytest.mark.parametrize("n,cap,threads", [(0, 5, 4), (1, 1, 4), (7, 9, 3), (100003, 100010, 16), (4096, 4096, 1)])
def test_allcore_exclusive_scan_matches_oracle(dtype, op, n, cap, threads):
    x = workloads.scan1d(dtype, capacity=cap, seed=50 + n)
    y = allcore.exclusive_scan(x, n, dtype, op, threads)
    want = oracle.exclusive_scan(x, n, dtype, op)
    if dtype == "f32" and op == "add":
        mag = np.concatenate([[0.0], np.cumsum(np.abs(x.numpy()[:n].astype(np.float64)))])[:n]
        assert np.all(np.abs(y[:n].astype(np.float64) - want.astype(np.float64)) <= 1e-5 * mag + 1e-6)
    else:
        assert np.array_equal(y[:n], want)


def test_allcore_exclusive_scan_wraps_like_the_oracle():
    x = torch.full((1000,), 2**31 - 7, dtype=torch.int32)
    assert np.array_equal(allcore.exclusive_scan(x, 1000, "i32", "add", 7), oracle.exclusive_scan(x, 1000, "i32", "add"))
