"""Seeded synthetic inputs for the scan library and its checker.

This module only draws random numbers and lays them out in the shapes of the
workloads below. It holds none of the scan arithmetic, so both the CUDA path
and the CPU oracle may use it without sharing any of the method.

Every tensor is drawn on the host with a fresh ``torch.Generator`` seeded with
the workload's seed, then cast to its storage dtype (bf16/f16 by torch's
round-to-nearest-even cast). Each tensor of a workload gets its own generator
seeded the same way, so one tensor's shape never shifts another's values.

Workloads (the shapes the pages bench on, sized for one GB300):

* ``rows_f32``      -- [1024, 4096] f32, iid uniform[-1, 1), seed 0
  (the bench shape of the metaltile-std ``mlx/scan.rs`` page, ``SCAN_SHAPES``).
* ``rows_half``     -- [8192, 8192] (exclusive) and [4096, 4099] (inclusive,
  ragged: n is not a multiple of 4 or 8) in bf16 and f16, iid N(0, 1), seed 1.
* ``rows_long``     -- [4, 2**24] f32, iid uniform[0, 1), seed 2; each row spans
  many tiles.
* ``scan1d``        -- 1-D capacity 2**28 with live count 2**28 - 12345:
  i32 uniform in [0, 15], i64 uniform in [0, 2**20), f32 uniform[-1, 1), seed 3.
* ``select``        -- f32 uniform[-1, 1) with u8 flags Bernoulli(p),
  p in {0.5, 0.01}, n = 2**28, seed 4.
"""
from __future__ import annotations

import torch

SEED_ROWS_F32 = 0
SEED_ROWS_HALF = 1
SEED_ROWS_LONG = 2
SEED_SCAN1D = 3
SEED_SELECT = 4

SCAN1D_CAPACITY = 1 << 28
SCAN1D_LIVE = (1 << 28) - 12345
SELECT_N = 1 << 28

_STORAGE = {
    "f32": torch.float32,
    "bf16": torch.bfloat16,
    "f16": torch.float16,
    "i32": torch.int32,
    "i64": torch.int64,
}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def uniform(shape, seed: int, lo: float, hi: float, dtype: str = "f32") -> torch.Tensor:
    """iid uniform[lo, hi) drawn in f32, then cast to the storage dtype."""
    u = torch.rand(shape, generator=generator(seed), dtype=torch.float32)
    if (lo, hi) == (-1.0, 1.0):
        x = u.mul_(2.0).sub_(1.0)
    elif (lo, hi) == (0.0, 1.0):
        x = u
    else:
        x = u.mul_(hi - lo).add_(lo)
    return x.to(_STORAGE[dtype])


def bits_uniform(shape, seed: int, dtype: str) -> torch.Tensor:
    """u32 / u64 values with every bit pattern equally likely (u64: the low
    63 bits uniform, the top bit set half the time)."""
    g = generator(seed)
    if dtype == "u32":
        return torch.randint(-(2**31), 2**31, shape, generator=g, dtype=torch.int32).view(torch.uint32)
    lo = torch.randint(-(2**62), 2**62, shape, generator=g, dtype=torch.int64)
    top = torch.randint(0, 2, shape, generator=g, dtype=torch.int64)
    return (lo ^ (top << 63)).view(torch.uint64)


def uniform64(shape, seed: int, lo: float, hi: float) -> torch.Tensor:
    """iid uniform[lo, hi) drawn directly in f64."""
    u = torch.rand(shape, generator=generator(seed), dtype=torch.float64)
    return u.mul_(hi - lo).add_(lo)


def normal(shape, seed: int, dtype: str = "f32") -> torch.Tensor:
    """iid N(0, 1) drawn in f32, then cast (round to nearest even) to storage."""
    x = torch.randn(shape, generator=generator(seed), dtype=torch.float32)
    return x.to(_STORAGE[dtype])


def randint(shape, seed: int, lo: int, hi_excl: int, dtype: str) -> torch.Tensor:
    """iid integers uniform in [lo, hi_excl)."""
    return torch.randint(lo, hi_excl, shape, generator=generator(seed),
                         dtype=_STORAGE[dtype])


def bernoulli_u8(n: int, p: float, seed: int) -> torch.Tensor:
    """Exactly-0/1 u8 flags, flag = (u < p) for u iid uniform[0, 1)."""
    u = torch.rand((n,), generator=generator(seed), dtype=torch.float32)
    return (u < p).to(torch.uint8)


def near_one(shape, seed: int, dtype: str = "f32", spread: float = 0.05) -> torch.Tensor:
    """Factors for product scans: a random sign times exp(u), u iid
    uniform[-spread, spread), drawn in f32 and cast to storage. The log of a
    prefix product is then a random walk with steps below `spread`, so
    products over tens of thousands of elements stay far from overflow and
    underflow in f32, bf16 and f16."""
    g = generator(seed)
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.int32).to(torch.float32).mul_(2.0).sub_(1.0)
    u = torch.rand(shape, generator=g, dtype=torch.float32).mul_(2.0 * spread).sub_(spread)
    return (sign * torch.exp(u)).to(_STORAGE[dtype])


def dyadic(shape, seed: int, dtype: str = "f32") -> torch.Tensor:
    """Values k/256 with integer |k| <= 255: exact in f32, bf16 and f16."""
    k = torch.randint(-255, 256, shape, generator=generator(seed), dtype=torch.int32)
    return (k.to(torch.float32) / 256.0).to(_STORAGE[dtype])


# ---- the named workloads ---------------------------------------------------

def rows_f32(rows: int = 1024, n: int = 4096, seed: int = SEED_ROWS_F32) -> torch.Tensor:
    return uniform((rows, n), seed, -1.0, 1.0, "f32")


def rows_half(rows: int, n: int, dtype: str, seed: int = SEED_ROWS_HALF) -> torch.Tensor:
    assert dtype in ("bf16", "f16")
    return normal((rows, n), seed, dtype)


def rows_long(rows: int = 4, n: int = 1 << 24, seed: int = SEED_ROWS_LONG) -> torch.Tensor:
    return uniform((rows, n), seed, 0.0, 1.0, "f32")


def scan1d(dtype: str, capacity: int = SCAN1D_CAPACITY, seed: int = SEED_SCAN1D) -> torch.Tensor:
    """The whole capacity is drawn; the live count is a separate argument."""
    if dtype == "i32":
        return randint((capacity,), seed, 0, 16, "i32")
    if dtype == "i64":
        return randint((capacity,), seed, 0, 1 << 20, "i64")
    if dtype == "f32":
        return uniform((capacity,), seed, -1.0, 1.0, "f32")
    # the other dtypes of the 1-D calls, drawn the same way (unsigned values
    # returned as their signed twins: the caller views them as unsigned)
    if dtype == "u32":
        return randint((capacity,), seed, 0, 16, "i32")
    if dtype == "u64":
        return randint((capacity,), seed, 0, 1 << 20, "i64")
    if dtype == "f64":
        return uniform64((capacity,), seed, -1.0, 1.0)
    raise ValueError(dtype)


def runs(n: int, mean_run: float, seed: int, key_dtype: str = "i32", val_dtype: str = "f32"):
    """(keys [n], values [n]) for reduce-by-key: run lengths geometric with
    the given mean, each run's key drawn from a small alphabet (so equal keys
    also recur in separate runs), values uniform[-1, 1) (f32) or integers in
    [-1000, 1000) (i32 / u32)."""
    g = generator(seed)
    starts = torch.rand((n,), generator=g) < (1.0 / mean_run)
    if n:
        starts[0] = True
    run_id = torch.cumsum(starts.to(torch.int64), 0) - 1
    alphabet = torch.randint(0, 64, (int(run_id[-1].item()) + 1 if n else 1,), generator=g,
                             dtype=torch.int64)
    k = alphabet[run_id] if n else torch.zeros((0,), dtype=torch.int64)
    keys = k.to(torch.float32) if key_dtype == "f32" else k.to(torch.int32)
    if key_dtype == "u32":
        keys = keys.view(torch.uint32)
    if val_dtype == "f32":
        vals = torch.rand((n,), generator=g, dtype=torch.float32).mul_(2.0).sub_(1.0)
    else:
        vals = torch.randint(-1000, 1000, (n,), generator=g, dtype=torch.int32)
        if val_dtype == "u32":
            vals = vals.view(torch.uint32)
    return keys, vals


def select_inputs(n: int = SELECT_N, p: float = 0.5, seed: int = SEED_SELECT):
    """(values f32 [n], flags u8 [n]); the flags use seed + 1 so p does not
    change the values."""
    vals = uniform((n,), seed, -1.0, 1.0, "f32")
    flags = bernoulli_u8(n, p, seed + 1)
    return vals, flags
