"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Each ``pin_*`` function raises AssertionError on a mismatch. They are run
directly by test_oracle_pins.py and, against builds of the oracle with a
planted mistake, by test_oracle_mutants.py (every planted mistake must make at
least one pin fail).

Kinds of pin used here:
  * values printed on the pages (tests/golden/, each file cites its passage);
  * closed forms (all-ones, arange, alternating signs);
  * invariants (exclusive = inclusive shifted right with the seed in front,
    exclusive[i] + x[i] = inclusive[i], the last prefix is the total);
  * brute force on tiny inputs with exact rational arithmetic;
  * special cases that reduce to a library routine (torch / numpy decoding,
    numpy's float64->float16 cast, cumulative min/max/sum);
  * an exact dyadic case where every association of the sum is exact.
"""
from __future__ import annotations

import bisect
from fractions import Fraction

import numpy as np
import torch

import oracle
from golden_io import load_all

I32_MAX, I32_MIN = 2**31 - 1, -(2**31)
I64_MAX, I64_MIN = 2**63 - 1, -(2**63)


# ---------------------------------------------------------------------------
# Tables of every finite bf16 / f16 value, decoded by torch / numpy (not by
# the oracle), for brute-force nearest-value rounding.
# ---------------------------------------------------------------------------
_TABLES = {}


def library_decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        t = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
        with np.errstate(invalid="ignore"):
            return t.to(torch.float32).numpy().astype(np.float64)
    return b.view(np.float16).astype(np.float64)


def _table(dtype):
    if dtype not in _TABLES:
        bits = np.arange(0, 0x7C00 if dtype == "f16" else 0x7F80, dtype=np.uint16)  # +0 .. max finite
        vals = library_decode(bits, dtype)
        order = np.argsort(vals, kind="stable")
        _TABLES[dtype] = (vals[order].tolist(), bits[order].tolist())
    return _TABLES[dtype]


def nearest_bits(x: float, dtype: str) -> int:
    """RN-even of a double to bf16/f16 by searching the table of values."""
    sign = 0x8000 if (np.signbit(x)) else 0
    a = abs(float(x))
    if np.isnan(a):
        raise ValueError("nan")
    vals, bits = _table(dtype)
    inf_bits = 0x7C00 if dtype == "f16" else 0x7F80
    if np.isinf(a):
        return sign | inf_bits
    mx = vals[-1]
    if a > mx:
        half = (mx - vals[-2]) / 2.0  # spacing at the top / 2 (exact)
        return sign | (inf_bits if a >= mx + half else bits[-1])
    i = bisect.bisect_left(vals, a)
    if vals[i] == a:
        return sign | bits[i]
    lo, hi = vals[i - 1], vals[i]
    mid = Fraction(lo) / 2 + Fraction(hi) / 2
    fa = Fraction(a)
    if fa < mid:
        return sign | bits[i - 1]
    if fa > mid:
        return sign | bits[i]
    return sign | (bits[i - 1] if bits[i - 1] % 2 == 0 else bits[i])


def rn_half_exact(values, dtype: str) -> np.ndarray:
    return np.array([nearest_bits(float(v), dtype) for v in values], dtype=np.uint16)


# ---------------------------------------------------------------------------
# Codecs
# ---------------------------------------------------------------------------

def pin_decode_all_patterns():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in ("bf16", "f16"):
        mine = oracle.decode_half(allbits, dt)
        ref = library_decode(allbits, dt)
        nan_m, nan_r = np.isnan(mine), np.isnan(ref)
        assert np.array_equal(nan_m, nan_r), dt
        ok = ~nan_r
        assert np.array_equal(mine[ok], ref[ok]), dt
        # signed zeros survive
        assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok])), dt


def pin_encode_round_trip_and_ties():
    for dt in ("bf16", "f16"):
        vals, bits = _table(dt)
        v = np.array(vals)
        b = np.array(bits, dtype=np.uint16)
        assert np.array_equal(oracle.encode_half(v, dt), b), dt
        assert np.array_equal(oracle.encode_half(-v, dt), b | 0x8000), dt
        # exact midpoints between neighbours: ties go to the even pattern
        mids = (v[:-1] + v[1:]) / 2.0
        even = np.where(b[:-1] % 2 == 0, b[:-1], b[1:])
        assert np.array_equal(oracle.encode_half(mids, dt), even), dt
        # just off the midpoint goes to the nearer neighbour
        up = np.nextafter(mids, np.inf)
        dn = np.nextafter(mids, -np.inf)
        assert np.array_equal(oracle.encode_half(up, dt), b[1:]), dt
        assert np.array_equal(oracle.encode_half(dn, dt), b[:-1]), dt
        # overflow: max + half spacing -> inf; just below -> max
        mx, spacing = v[-1], v[-1] - v[-2]
        inf_bits = 0x7C00 if dt == "f16" else 0x7F80
        enc = oracle.encode_half(np.array([mx + spacing / 2, np.nextafter(mx + spacing / 2, 0),
                                           np.inf, -np.inf, 1e300]), dt)
        assert list(enc) == [inf_bits, b[-1], inf_bits, inf_bits | 0x8000, inf_bits], dt
        # NaN is quieted
        enc_nan = int(oracle.encode_half(np.array([np.nan]), dt)[0])
        assert (enc_nan & inf_bits) == inf_bits and (enc_nan & 0x03FF if dt == "f16" else enc_nan & 0x7F) != 0


def pin_encode_random_doubles():
    rng = np.random.default_rng(1234)
    for dt, (emin, emax) in (("bf16", (-140, 128)), ("f16", (-27, 16))):
        m = rng.uniform(1.0, 2.0, 20000)
        e = rng.integers(emin, emax + 1, 20000)
        x = np.ldexp(m, e) * np.where(rng.random(20000) < 0.5, -1.0, 1.0)
        got = oracle.encode_half(x, dt)
        want = rn_half_exact(x, dt)
        assert np.array_equal(got, want), dt
    # numpy's float64 -> float16 cast is a library routine for the same rounding
    x = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-27, 16, 20000))
    assert np.array_equal(oracle.encode_half(x, "f16"), x.astype(np.float16).view(np.uint16))


def pin_ulp():
    rng = np.random.default_rng(7)
    for dt, npt in (("f32", np.float32), ("f16", np.float16)):
        x = np.ldexp(rng.uniform(1, 2, 200), rng.integers(-30, 15, 200)).astype(npt)
        for v in x:
            assert oracle.ulp(float(v), dt) == float(np.spacing(npt(abs(v)))), (dt, v)
    # bf16: the gap to the next pattern up, from the library-decoded table
    vals, _ = _table("bf16")
    for i in (0, 1, 5, 127, 128, 129, 5000, 16000, 32000):
        assert oracle.ulp(vals[i], "bf16") == vals[i + 1] - vals[i] or i == 0
    assert oracle.ulp(0.0, "bf16") == vals[1]
    # the vectorised numpy form agrees with the C function
    for dt in ("f32", "bf16", "f16"):
        v = np.ldexp(rng.uniform(1, 2, 300), rng.integers(-150, 20, 300))
        v[:5] = 0.0
        assert np.array_equal(oracle.ulp_array(v, dt), np.array([oracle.ulp(t, dt) for t in v])), dt


# ---------------------------------------------------------------------------
# Row-wise scan
# ---------------------------------------------------------------------------

def _f32(a):
    return torch.tensor(np.asarray(a, dtype=np.float32))


def pin_rows_golden_order():
    g = load_all()["tile_inclusive_order"]
    for s in ("a", "b"):
        x = _f32([g["x_" + s]])
        out = oracle.scan_rows(x, "f32", True)
        assert out[0].tolist() == [float(v) for v in g["inclusive_" + s]], s


def pin_rows_closed_forms():
    rows, n = 3, 1000
    ones = torch.ones(rows, n)
    inc = oracle.scan_rows(ones, "f32", True)
    exc = oracle.scan_rows(ones, "f32", False)
    i = np.arange(n, dtype=np.float64)
    assert np.array_equal(inc, np.broadcast_to(i + 1, (rows, n)).astype(np.float32))
    assert np.array_equal(exc, np.broadcast_to(i, (rows, n)).astype(np.float32))
    ar = torch.arange(n, dtype=torch.float32).repeat(rows, 1) * torch.tensor([[1.0], [2.0], [-1.0]])
    inc = oracle.scan_rows(ar, "f32", True)
    tri = i * (i + 1) / 2
    assert np.array_equal(inc, np.stack([tri, 2 * tri, -tri]).astype(np.float32))
    # alternating signs in f16: 1, 0, 1, 0, ...
    alt = torch.tensor([[(-1.0) ** k for k in range(257)]], dtype=torch.float16)
    inc = oracle.scan_rows(alt, "f16", True)
    assert np.array_equal(library_decode(inc[0], "f16"), np.array([1.0 - (k % 2) for k in range(257)]))
    # bf16 ones: the exact prefix i+1 rounded to nearest even in bf16
    n2 = 700
    inc = oracle.scan_rows(torch.ones(2, n2, dtype=torch.bfloat16), "bf16", True)
    exc = oracle.scan_rows(torch.ones(2, n2, dtype=torch.bfloat16), "bf16", False)
    assert np.array_equal(inc[1], rn_half_exact(np.arange(1, n2 + 1), "bf16"))
    assert np.array_equal(exc[0], rn_half_exact(np.arange(0, n2), "bf16"))
    assert int(exc[0, 0]) == 0  # exclusive out[0] = 0 (scan.rs module doc)


def pin_rows_brute_force_exact():
    """Tiny rows, each prefix recomputed independently with Fractions."""
    rng = np.random.default_rng(99)
    for dt in ("f32", "bf16", "f16"):
        for n in (1, 2, 3, 7, 31, 33, 64):
            # multiples of 2^-12 in [-4, 4]: fp64 sums of <= 64 terms are exact
            k = rng.integers(-(2**14), 2**14, size=(3, n))
            x = torch.tensor(k / 4096.0, dtype=torch.float32).to(
                {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dt])
            xd = x.to(torch.float64).numpy()
            for inclusive in (True, False):
                out, p64, m64 = oracle.scan_rows(x, dt, inclusive, want_f64=True)
                for r in range(3):
                    for i in range(n):
                        hi = i + 1 if inclusive else i
                        exact = sum((Fraction(float(v)) for v in xd[r, :hi]), Fraction(0))
                        assert Fraction(float(p64[r, i])) == exact, (dt, n, r, i)
                        mag = sum(abs(Fraction(float(v))) for v in xd[r, :i + 1])
                        assert Fraction(float(m64[r, i])) == mag
                        if dt == "f32":
                            assert out[r, i] == np.float32(float(exact))
                        else:
                            assert int(out[r, i]) == nearest_bits(float(exact), dt), (dt, r, i)


def pin_rows_invariants_and_library():
    x = torch.rand(5, 3001, generator=torch.Generator().manual_seed(5)) * 2 - 1
    _, inc, mag = oracle.scan_rows(x, "f32", True, want_f64=True)
    _, exc, _ = oracle.scan_rows(x, "f32", False, want_f64=True)
    xd = x.double().numpy()
    assert np.all(exc[:, 0] == 0.0)
    assert np.array_equal(exc[:, 1:], inc[:, :-1])          # shift right by one
    assert np.array_equal(exc + xd, inc)                     # exclusive + x = inclusive
    assert np.array_equal(inc, torch.cumsum(x.double(), dim=1).numpy())  # library cumsum
    assert np.allclose(mag[:, -1], np.abs(xd).sum(axis=1), rtol=1e-13, atol=0)
    tot = np.array([float(sum(Fraction(float(v)) for v in row)) for row in xd])
    assert np.allclose(inc[:, -1], tot, rtol=0, atol=1e-12)  # last prefix = total


def pin_rows_dyadic_exact():
    """k/256 inputs, n = 2^15: every partial sum is exact in f32, so the
    rounded output is RN_T(exact prefix) whatever the summation order."""
    rows, n = 2, 1 << 15
    k = torch.randint(-255, 256, (rows, n), generator=torch.Generator().manual_seed(11))
    pre = torch.cumsum(k.to(torch.int64), dim=1).numpy()     # exact integer prefixes
    for dt, tdt in (("f32", torch.float32), ("bf16", torch.bfloat16), ("f16", torch.float16)):
        x = (k.to(torch.float32) / 256.0).to(tdt)
        for inclusive in (True, False):
            num = pre if inclusive else np.concatenate([np.zeros((rows, 1), np.int64), pre[:, :-1]], 1)
            exact = num / 256.0
            out = oracle.scan_rows(x, dt, inclusive)
            if dt == "f32":
                assert np.array_equal(out, exact.astype(np.float32))
            else:
                sub = slice(0, n, 37)  # table search is slow in Python: a stride sample
                want = rn_half_exact(exact[:, sub].ravel(), dt).reshape(rows, -1)
                assert np.array_equal(out[:, sub], want), dt


def pin_rows_empty():
    for shape in ((0, 5), (3, 0), (0, 0)):
        out = oracle.scan_rows(torch.zeros(shape), "f32", True)
        assert out.shape == shape


# ---------------------------------------------------------------------------
# Device-wide exclusive scan
# ---------------------------------------------------------------------------

_NP = {"i32": np.int32, "i64": np.int64, "f32": np.float32}
_IDENT = {("i32", "add"): 0, ("i32", "min"): I32_MAX, ("i32", "max"): I32_MIN,
          ("i64", "add"): 0, ("i64", "min"): I64_MAX, ("i64", "max"): I64_MIN,
          ("f32", "add"): 0.0, ("f32", "min"): np.inf, ("f32", "max"): -np.inf}


def pin_scan_golden():
    g = load_all()
    ex = g["algos_exclusive_scan_add_i32"]
    for dt in ("i32", "i64", "f32"):
        arr = np.array(ex["arr"], dtype=_NP[dt])
        out = oracle.exclusive_scan(arr, len(arr), dt, "add")
        assert out.tolist() == ex["exclusive"], dt
    mm = g["algos_exclusive_scan_minmax_i32"]
    arr = np.array(mm["arr"], dtype=np.int32)
    for op in ("min", "max"):
        assert oracle.exclusive_scan(arr, len(arr), "i32", op).tolist() == mm[op], op
    red = g["algos_reduce_i32"]
    ext = np.array(red["arr"] + [0], dtype=np.int32)  # one more slot: its prefix is the reduction
    for op in ("add", "min", "max"):
        assert int(oracle.exclusive_scan(ext, len(ext), "i32", op)[-1]) == red[op], op


def pin_scan_identities():
    for (dt, op), ident in _IDENT.items():
        arr = np.array([5, 7], dtype=_NP[dt])
        out = oracle.exclusive_scan(arr, 1, dt, op)
        assert out.shape == (1,) and out[0] == ident, (dt, op)
        assert oracle.exclusive_scan(arr, 0, dt, op).shape == (0,)
    x = np.array([np.inf, -np.inf, 0.5], dtype=np.float32)
    assert oracle.exclusive_scan(x, 3, "f32", "min").tolist() == [np.inf, np.inf, -np.inf]
    assert oracle.exclusive_scan(x, 3, "f32", "max").tolist() == [-np.inf, np.inf, np.inf]


def pin_scan_wrap():
    a = np.array([I32_MAX, 1, 5], dtype=np.int32)
    assert oracle.exclusive_scan(a, 3, "i32", "add").tolist() == [0, I32_MAX, I32_MIN]
    b = np.array([I64_MAX, 1, 0], dtype=np.int64)
    assert oracle.exclusive_scan(b, 3, "i64", "add").tolist() == [0, I64_MAX, I64_MIN]


def pin_scan_library():
    rng = np.random.default_rng(3)
    n = 20000
    for dt in ("i32", "i64", "f32"):
        if dt == "i32":
            x = rng.integers(-(2**31), 2**31, n, dtype=np.int64).astype(np.int32)
        elif dt == "i64":
            x = rng.integers(-(2**62), 2**62, n, dtype=np.int64)
        else:
            x = rng.uniform(-1, 1, n).astype(np.float32)
        for op, acc in (("min", np.minimum.accumulate), ("max", np.maximum.accumulate)):
            want = np.concatenate([[_IDENT[(dt, op)]], acc(x)[:-1]]).astype(_NP[dt])
            assert np.array_equal(oracle.exclusive_scan(x, n, dt, op), want), (dt, op)
        if dt == "i32":
            s = np.cumsum(x.astype(np.int64)) & 0xFFFFFFFF
            want = np.concatenate([[0], s[:-1]]).astype(np.uint32).view(np.int32)
            assert np.array_equal(oracle.exclusive_scan(x, n, dt, "add"), want)
        elif dt == "i64":
            with np.errstate(over="ignore"):
                want = np.concatenate([[0], np.cumsum(x)[:-1]])
            assert np.array_equal(oracle.exclusive_scan(x, n, dt, "add"), want)
        else:
            out, p64, mag = oracle.exclusive_scan(x, n, dt, "add", want_f64=True)
            want = np.concatenate([[0.0], np.cumsum(x.astype(np.float64))[:-1]])
            assert np.array_equal(p64, want)
            assert np.array_equal(out, want.astype(np.float32))
            assert np.allclose(mag, np.cumsum(np.abs(x.astype(np.float64))), rtol=1e-13, atol=0)


def pin_scan_brute_force():
    rng = np.random.default_rng(17)
    for n in (1, 2, 5, 32, 33, 64):
        for dt in ("i32", "i64", "f32"):
            if dt == "f32":
                x = (rng.integers(-4096, 4096, n) / 1024.0).astype(np.float32)
            else:
                x = rng.integers(-1000, 1000, n).astype(_NP[dt])
            for op in ("add", "min", "max"):
                out = oracle.exclusive_scan(x, n, dt, op)
                for i in range(n):
                    head = [x[j].item() for j in range(i)]
                    if op == "add":
                        want = sum((Fraction(v) for v in head), Fraction(0))
                    elif op == "min":
                        want = min(head, default=_IDENT[(dt, op)])
                    else:
                        want = max(head, default=_IDENT[(dt, op)])
                    got = out[i].item()
                    if op == "add":
                        assert Fraction(got) == want, (n, dt, op, i)
                    else:
                        assert got == want, (n, dt, op, i)


def pin_inclusive_golden():
    g = load_all()
    ex = g["algos_inclusive_scan_add_i32"]
    tile = g["tile_inclusive_order"]
    for dt in ("i32", "i64", "f32"):
        arr = np.array(ex["arr"], dtype=_NP[dt])
        assert oracle.inclusive_scan(arr, len(arr), dt, "add").tolist() == ex["inclusive"], dt
        assert oracle.inclusive_scan(arr, len(arr), dt, "min").tolist() == ex["inclusive_min"], dt
        assert oracle.inclusive_scan(arr, len(arr), dt, "max").tolist() == ex["inclusive_max"], dt
        for a, b in (("x_a", "inclusive_a"), ("x_b", "inclusive_b")):
            x = np.array(tile[a], dtype=_NP[dt])
            assert oracle.inclusive_scan(x, len(x), dt, "add").tolist() == tile[b], (dt, a)


def pin_inclusive_brute_force():
    rng = np.random.default_rng(29)
    for n in (0, 1, 2, 5, 33, 64):
        for dt in ("i32", "i64", "f32"):
            if dt == "f32":
                x = (rng.integers(-4096, 4096, n) / 1024.0).astype(np.float32)
            else:
                x = rng.integers(-1000, 1000, n).astype(_NP[dt])
            for op in ("add", "min", "max"):
                out = oracle.inclusive_scan(x, n, dt, op)
                assert out.shape == (n,)
                for i in range(n):
                    head = [x[j].item() for j in range(i + 1)]
                    if op == "add":
                        assert Fraction(out[i].item()) == sum(Fraction(v) for v in head), (n, dt, i)
                    elif op == "min":
                        assert out[i].item() == min(head), (n, dt, i)
                    else:
                        assert out[i].item() == max(head), (n, dt, i)


def pin_inclusive_library():
    rng = np.random.default_rng(31)
    n = 20000
    for dt in ("i32", "i64", "f32"):
        if dt == "i32":
            x = rng.integers(-(2**31), 2**31, n, dtype=np.int64).astype(np.int32)
        elif dt == "i64":
            x = rng.integers(-(2**62), 2**62, n, dtype=np.int64)
        else:
            x = rng.uniform(-1, 1, n).astype(np.float32)
        assert np.array_equal(oracle.inclusive_scan(x, n, dt, "min"), np.minimum.accumulate(x))
        assert np.array_equal(oracle.inclusive_scan(x, n, dt, "max"), np.maximum.accumulate(x))
        if dt == "i32":
            want = (np.cumsum(x.astype(np.int64)) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
            assert np.array_equal(oracle.inclusive_scan(x, n, dt, "add"), want)
        elif dt == "i64":
            with np.errstate(over="ignore"):
                want = np.cumsum(x)
            assert np.array_equal(oracle.inclusive_scan(x, n, dt, "add"), want)
        else:
            out, p64, mag = oracle.inclusive_scan(x, n, dt, "add", want_f64=True)
            want = np.cumsum(x.astype(np.float64))
            assert np.array_equal(p64, want)
            assert np.array_equal(out, want.astype(np.float32))
            assert np.allclose(mag, np.cumsum(np.abs(x.astype(np.float64))), rtol=1e-13, atol=0)


def pin_reduce_golden_and_identities():
    red = load_all()["algos_reduce_i32"]
    for dt in ("i32", "i64", "f32"):
        arr = np.array(red["arr"], dtype=_NP[dt])
        for op in ("add", "min", "max"):
            assert oracle.reduce(arr, len(arr), dt, op) == red[op], (dt, op)
            assert oracle.reduce(arr, 0, dt, op) == _IDENT[(dt, op)], (dt, op)
            assert oracle.reduce(arr, 1, dt, op) == red["arr"][0], (dt, op)
    a = np.array([I32_MAX, 1], dtype=np.int32)
    assert oracle.reduce(a, 2, "i32", "add") == I32_MIN  # wraps
    b = np.array([I64_MAX, 1], dtype=np.int64)
    assert oracle.reduce(b, 2, "i64", "add") == I64_MIN


def pin_reduce_library():
    rng = np.random.default_rng(37)
    for n in (1, 7, 1000, 50001):
        for dt in ("i32", "i64", "f32"):
            if dt == "i32":
                x = rng.integers(-(2**31), 2**31, n, dtype=np.int64).astype(np.int32)
            elif dt == "i64":
                x = rng.integers(-(2**62), 2**62, n, dtype=np.int64)
            else:
                x = rng.uniform(-1, 1, n).astype(np.float32)
            assert oracle.reduce(x, n, dt, "min") == x.min()
            assert oracle.reduce(x, n, dt, "max") == x.max()
            if dt == "i32":
                want = int(x.astype(np.int64).sum()) & 0xFFFFFFFF
                want = want - 2**32 if want >= 2**31 else want
                assert int(oracle.reduce(x, n, dt, "add")) == want
            elif dt == "i64":
                want = (int(sum(int(v) for v in x)) + 2**63) % 2**64 - 2**63
                assert int(oracle.reduce(x, n, dt, "add")) == want
            else:
                r, s64, m64 = oracle.reduce(x, n, dt, "add", want_f64=True)
                seq = np.cumsum(x.astype(np.float64))[-1]  # the same left-to-right order
                assert s64 == seq and r == np.float32(seq)
                assert abs(m64 - np.abs(x.astype(np.float64)).sum()) <= 1e-12 * m64


def pin_reduce_signed_zero_ties():
    """min/max keep the earliest of equal values: the sign of a zero result
    is that of the first zero."""
    pz, nz = np.float32(0.0), np.float32(-0.0)
    for first, second in ((pz, nz), (nz, pz)):
        x = np.array([1.0, first, 2.0, second], dtype=np.float32)
        for op in ("min",):
            r = oracle.reduce(x, 4, "f32", op)
            assert r == 0 and np.signbit(r) == np.signbit(first)
        y = np.array([-1.0, first, -2.0, second], dtype=np.float32)
        r = oracle.reduce(y, 4, "f32", "max")
        assert r == 0 and np.signbit(r) == np.signbit(first)
        inc = oracle.inclusive_scan(x, 4, "f32", "min")
        assert np.signbit(inc[3]) == np.signbit(first)


# ---------------------------------------------------------------------------
# The unsigned and f64 dtypes of the 1-D calls
# ---------------------------------------------------------------------------
U32_MAX, U64_MAX = 2**32 - 1, 2**64 - 1
_NPX = {"u32": np.uint32, "u64": np.uint64, "f64": np.float64}
_IDX = {("u32", "add"): 0, ("u32", "min"): U32_MAX, ("u32", "max"): 0,
        ("u64", "add"): 0, ("u64", "min"): U64_MAX, ("u64", "max"): 0,
        ("f64", "add"): 0.0, ("f64", "min"): np.inf, ("f64", "max"): -np.inf}


def pin_ext_golden():
    g = load_all()
    ex = g["algos_exclusive_scan_add_i32"]
    inc = g["algos_inclusive_scan_add_i32"]
    mm = g["algos_exclusive_scan_minmax_i32"]
    red = g["algos_reduce_i32"]
    for dt in ("u32", "u64", "f64"):
        arr = np.array(ex["arr"], dtype=_NPX[dt])
        assert oracle.exclusive_scan(arr, len(arr), dt, "add").tolist() == ex["exclusive"], dt
        assert oracle.inclusive_scan(arr, len(arr), dt, "add").tolist() == inc["inclusive"], dt
        for op in ("min", "max"):
            got = oracle.exclusive_scan(np.array(mm["arr"], dtype=_NPX[dt]), len(mm["arr"]), dt, op)
            want = [(_IDX[(dt, op)] if i == 0 else v) for i, v in enumerate(mm[op])]
            assert got.tolist() == want, (dt, op)
        for op in ("add", "min", "max"):
            assert oracle.reduce(arr, len(arr), dt, op) == red[op], (dt, op)
            assert oracle.reduce(arr, 0, dt, op) == _IDX[(dt, op)], (dt, op)


def pin_ext_unsigned_order_and_wrap():
    a = np.array([1, 2**31 + 5, 3, U32_MAX], dtype=np.uint32)
    assert oracle.inclusive_scan(a, 4, "u32", "max").tolist() == [1, 2**31 + 5, 2**31 + 5, U32_MAX]
    assert oracle.inclusive_scan(a, 4, "u32", "min").tolist() == [1, 1, 1, 1]
    assert oracle.exclusive_scan(a, 4, "u32", "add").tolist() == [0, 1, 2**31 + 6, 2**31 + 9]
    assert oracle.reduce(a, 4, "u32", "add") == (1 + 2**31 + 5 + 3 + U32_MAX) % 2**32
    b = np.array([2**63 + 7, 1, U64_MAX], dtype=np.uint64)
    assert oracle.inclusive_scan(b, 3, "u64", "max").tolist() == [2**63 + 7, 2**63 + 7, U64_MAX]
    assert oracle.inclusive_scan(b, 3, "u64", "min").tolist() == [2**63 + 7, 1, 1]
    assert oracle.inclusive_scan(b, 3, "u64", "add").tolist() == [2**63 + 7, 2**63 + 8, 2**63 + 7]
    assert oracle.reduce(b, 3, "u64", "min") == 1


def pin_ext_library():
    rng = np.random.default_rng(47)
    n = 20000
    for dt in ("u32", "u64", "f64"):
        if dt == "u32":
            x = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
        elif dt == "u64":
            x = rng.integers(0, 2**63, n, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
        else:
            x = rng.uniform(-1, 1, n)
        assert np.array_equal(oracle.inclusive_scan(x, n, dt, "min"), np.minimum.accumulate(x))
        assert np.array_equal(oracle.inclusive_scan(x, n, dt, "max"), np.maximum.accumulate(x))
        assert oracle.reduce(x, n, dt, "min") == x.min() and oracle.reduce(x, n, dt, "max") == x.max()
        if dt != "f64":
            with np.errstate(over="ignore"):
                want = np.cumsum(x, dtype=x.dtype)  # numpy wraps unsigned sums
            assert np.array_equal(oracle.inclusive_scan(x, n, dt, "add"), want)
            assert oracle.reduce(x, n, dt, "add") == want[-1]


def pin_ext_f64_signed_zero_ties():
    for first in (0.0, -0.0):
        second = -0.0 if not np.signbit(first) else 0.0
        x = np.array([1.0, first, 2.0, second])
        r = oracle.reduce(x, 4, "f64", "min")
        assert r == 0 and np.signbit(r) == np.signbit(first)
        y = np.array([-1.0, first, -2.0, second])
        r = oracle.reduce(y, 4, "f64", "max")
        assert r == 0 and np.signbit(r) == np.signbit(first)
        inc = oracle.inclusive_scan(y, 4, "f64", "max")
        assert np.signbit(inc[3]) == np.signbit(first)


def pin_ext_f64_sums():
    """Dyadic f64 inputs: every prefix is exact, so the oracle's prefix is
    the exact one; random inputs: each prefix within one ulp of the
    correctly rounded prefix (math.fsum)."""
    import math
    rng = np.random.default_rng(53)
    x = rng.integers(-2**20, 2**20, 5000) / 1024.0
    out, p, mag = oracle.inclusive_scan(x, 5000, "f64", "add", want_f64=True)
    assert np.array_equal(p, np.cumsum(x)) and np.array_equal(out, p)
    assert np.array_equal(mag, np.cumsum(np.abs(x)))
    ex = oracle.exclusive_scan(x, 5000, "f64", "add")
    assert ex[0] == 0.0 and np.array_equal(ex[1:], p[:-1])
    y = rng.uniform(-1, 1, 2000) * 10.0 ** rng.integers(-8, 9, 2000)
    got = oracle.inclusive_scan(y, 2000, "f64", "add")
    for i in range(0, 2000, 97):
        want = math.fsum(y[: i + 1])
        assert abs(got[i] - want) <= np.spacing(abs(want)) + 1e-300, i
    r, s64, m64 = oracle.reduce(y, 2000, "f64", "add", want_f64=True)
    assert abs(r - math.fsum(y)) <= np.spacing(abs(math.fsum(y)))


# ---------------------------------------------------------------------------
# Row scans with prod / max / min
# ---------------------------------------------------------------------------

def _num(tok):
    return float(tok) if isinstance(tok, str) else float(tok)


def pin_rows_op_golden():
    g = load_all()["scanrs_multi_op"]
    x = np.array([g["x"]], dtype=np.float32)
    for op in ("prod", "max", "min"):
        for kind in ("inclusive", "exclusive"):
            want = [_num(t) for t in g[f"{op}_{kind}"]]
            opn = "mul" if op == "prod" else op
            for dt in ("f32", "bf16", "f16"):
                xs = torch.from_numpy(x).to(torch.bfloat16 if dt == "bf16" else torch.float16) \
                    if dt != "f32" else torch.from_numpy(x)
                out = oracle.scan_rows_op(xs, dt, opn, kind == "inclusive")
                if dt == "f32":
                    got, exp = out[0].astype(np.float64), [float(np.float32(w)) for w in want]
                else:  # the page's exact values rounded to the storage type by table search
                    got = library_decode(out[0], dt)
                    exp = [w if np.isinf(w) else float(library_decode(
                        np.array([nearest_bits(w, dt)], dtype=np.uint16), dt)[0]) for w in want]
                assert got.tolist() == exp, (op, kind, dt)


def pin_rows_op_brute_force():
    """Small-integer rows: every prefix product is an exact integer below
    2^24, so the rounded prefix is exact in every storage type up to 2048
    (bf16: 256) and is checked against exact integer arithmetic."""
    rng = np.random.default_rng(41)
    for dt, lim in (("f32", 1 << 24), ("f16", 2048), ("bf16", 256)):
        for n in (1, 2, 7, 33):
            x = rng.choice([-2.0, -1.0, 1.0, 2.0], size=(3, n)).astype(np.float32)
            xs = torch.from_numpy(x) if dt == "f32" else torch.from_numpy(x).to(
                torch.bfloat16 if dt == "bf16" else torch.float16)
            for inclusive in (True, False):
                for op in ("mul", "min", "max"):
                    out = oracle.scan_rows_op(xs, dt, op, inclusive)
                    got = out.astype(np.float64) if dt == "f32" else library_decode(out, dt)
                    for r in range(3):
                        acc = {"mul": 1, "min": float("inf"), "max": float("-inf")}[op]
                        for i in range(n):
                            v = int(x[r, i])
                            nxt = acc * v if op == "mul" else (min(acc, v) if op == "min" else max(acc, v))
                            want = nxt if inclusive else acc
                            if op == "mul" and abs(want) > lim:
                                acc = nxt
                                continue
                            assert got[r, i] == want, (dt, op, inclusive, r, i)
                            acc = nxt


def pin_rows_op_library():
    rng = np.random.default_rng(43)
    x = (rng.choice([-1.0, 1.0], size=(4, 3000)) *
         np.exp(rng.uniform(-0.05, 0.05, size=(4, 3000)))).astype(np.float32)
    x64 = x.astype(np.float64)
    for inclusive in (True, False):
        for op, acc, seed in (("mul", np.multiply.accumulate, 1.0),
                              ("min", np.minimum.accumulate, np.inf),
                              ("max", np.maximum.accumulate, -np.inf),
                              ("add", np.add.accumulate, 0.0)):
            out, p64 = oracle.scan_rows_op(x, "f32", op, inclusive, want_f64=True)
            want = acc(x64, axis=1)
            if not inclusive:
                want = np.concatenate([np.full((4, 1), seed), want[:, :-1]], axis=1)
            assert np.array_equal(p64, want), (op, inclusive)
            assert np.array_equal(out, want.astype(np.float32)), (op, inclusive)


def pin_rows_op_signed_zero_ties():
    pz, nz = 0.0, -0.0
    for first in (pz, nz):
        second = nz if first == pz and not np.signbit(first) else pz
        x = np.array([[1.0, first, second, 3.0]], dtype=np.float32)
        out = oracle.scan_rows_op(x, "f32", "min", True)
        assert out[0, 1] == 0 and np.signbit(out[0, 2]) == np.signbit(first)
        y = np.array([[-1.0, first, second, -3.0]], dtype=np.float32)
        out = oracle.scan_rows_op(y, "f32", "max", True)
        assert out[0, 3] == 0 and np.signbit(out[0, 3]) == np.signbit(first)


# ---------------------------------------------------------------------------
# Select
# ---------------------------------------------------------------------------

def pin_select_golden():
    g = load_all()["algos_select_i32"]
    arr = np.array(g["arr"], dtype=np.int32)
    flags = np.array(g["flags"], dtype=np.uint8)
    out, k = oracle.select(arr, flags, len(arr))
    assert k == g["num_out"]
    assert out.view(np.int32).tolist() == g["out"]


def pin_select_brute_force():
    rng = np.random.default_rng(23)
    for n in (0, 1, 2, 17, 300, 5000):
        for p in (0.0, 0.01, 0.5, 1.0):
            bits = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)  # any bit pattern
            flags = (rng.random(n) < p).astype(np.uint8)
            out, k = oracle.select(bits, flags, n)
            want = [int(b) for b, f in zip(bits, flags) if f == 1]
            assert k == int(flags.sum()) == len(want)
            assert out.tolist() == want


def pin_select_wide():
    g = load_all()["algos_select_i32"]
    for eb, dt in ((4, np.int32), (8, np.int64)):
        arr = np.array(g["arr"], dtype=dt)
        flags = np.array(g["flags"], dtype=np.uint8)
        out, k = oracle.select_wide(arr, flags, len(arr), eb)
        assert k == g["num_out"] and out.view(dt).tolist() == g["out"], eb
    rng = np.random.default_rng(59)
    for n in (0, 1, 300, 5000):
        bits = rng.integers(0, 2**63, n, dtype=np.uint64) * np.uint64(2) + rng.integers(0, 2, n, dtype=np.uint64)
        flags = (rng.random(n) < 0.3).astype(np.uint8)
        out, k = oracle.select_wide(bits, flags, n, 8)
        want = [int(b) for b, f in zip(bits, flags) if f == 1]
        assert k == len(want) and out.tolist() == want


def pin_select_struct_elements():
    """Struct elements ([algos] select: the scatter copies each field): a
    compaction of structs equals the compaction of each field column with
    the same flags, and a plain Python filter on tiny inputs."""
    rng = np.random.default_rng(61)
    for words in (3, 4, 6, 9, 64):  # 12- to 256-byte structs of 32-bit fields
        for n in (0, 1, 7, 300, 2000):
            arr = rng.integers(0, 2**32, (n, words), dtype=np.uint64).astype(np.uint32)
            flags = (rng.random(n) < 0.4).astype(np.uint8)
            out, k = oracle.select_wide(arr, flags, n, 4 * words)
            assert k == int(flags.sum())
            got = out.view(np.uint32).reshape(k, words)
            for w in range(words):
                col, kc = oracle.select(np.ascontiguousarray(arr[:, w]), flags, n)
                assert kc == k and np.array_equal(got[:, w], col), (words, n, w)
            if n <= 7:
                want = [list(map(int, arr[i])) for i in range(n) if flags[i] == 1]
                assert got.tolist() == want
    # an element size that is not a multiple of 4 (3-byte records) by brute force
    rec = rng.integers(0, 256, (50, 3), dtype=np.uint8)
    flags = (rng.random(50) < 0.5).astype(np.uint8)
    out, k = oracle.select_wide(rec, flags, 50, 3)
    assert out.tolist() == [list(map(int, rec[i])) for i in range(50) if flags[i] == 1]


# ---------------------------------------------------------------------------
# Reduce by key
# ---------------------------------------------------------------------------

def pin_reduce_by_key_golden():
    g = load_all()["algos_reduce_by_key_add_i32"]
    for kd, vd in (("i32", "i32"), ("u32", "u32"), ("f32", "f32"), ("i32", "f32")):
        keys = np.array(g["keys"], dtype={"i32": np.int32, "u32": np.uint32, "f32": np.float32}[kd])
        vals = np.array(g["values"], dtype={"i32": np.int32, "u32": np.uint32, "f32": np.float32}[vd])
        ko, vo, r = oracle.reduce_by_key_add(keys, vals, len(keys), kd, vd)
        assert r == g["num_runs"] and ko.tolist() == g["keys_out"] and vo.tolist() == g["values_out"]


def pin_reduce_by_key_brute_force():
    """Runs found by an independent scan with itertools.groupby-style logic."""
    rng = np.random.default_rng(67)
    for n in (0, 1, 2, 9, 300, 5000):
        keys = rng.integers(0, 4, n).astype(np.int32)  # small alphabet: long and short runs
        vals = rng.integers(-1000, 1000, n).astype(np.int32)
        ko, vo, r = oracle.reduce_by_key_add(keys, vals, n, "i32", "i32")
        want_k, want_v = [], []
        for i in range(n):
            if i == 0 or keys[i] != keys[i - 1]:
                want_k.append(int(keys[i]))
                want_v.append(0)
            want_v[-1] += int(vals[i])
        assert r == len(want_k) and ko.tolist() == want_k and vo.tolist() == want_v, n
        fv = (rng.integers(-4096, 4096, n) / 256.0).astype(np.float32)  # exact partial sums
        ko, vo, r, s64, m64 = oracle.reduce_by_key_add(keys, fv, n, "i32", "f32", want_f64=True)
        j = -1
        sums, mags = [], []
        for i in range(n):
            if i == 0 or keys[i] != keys[i - 1]:
                sums.append(Fraction(0))
                mags.append(Fraction(0))
            sums[-1] += Fraction(float(fv[i]))
            mags[-1] += abs(Fraction(float(fv[i])))
        assert [Fraction(float(x)) for x in vo] == sums and [Fraction(x) for x in s64] == sums
        assert [Fraction(x) for x in m64] == mags


def pin_reduce_by_key_float_keys_and_wrap():
    nan = np.float32("nan")
    keys = np.array([1.0, nan, nan, 0.0, -0.0, 2.0, 2.0, 1.0], dtype=np.float32)
    vals = np.arange(1, 9, dtype=np.int32)
    ko, vo, r = oracle.reduce_by_key_add(keys, vals, 8, "f32", "i32")
    assert r == 6  # 1 | nan | nan | (0, -0) | (2, 2) | 1
    assert vo.tolist() == [1, 2, 3, 4 + 5, 6 + 7, 8]
    assert np.isnan(ko[1]) and np.isnan(ko[2]) and ko[3] == 0 and not np.signbit(ko[3])
    u = np.array([7, 7, 7], dtype=np.uint32)
    w = np.array([2**32 - 1, 2, 2**31], dtype=np.uint32)
    _, vo, r = oracle.reduce_by_key_add(u, w, 3, "u32", "u32")
    assert r == 1 and int(vo[0]) == (2**32 - 1 + 2 + 2**31) % 2**32


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
