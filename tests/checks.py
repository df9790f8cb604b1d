"""Comparison of CUDA-path outputs with the CPU oracle.

Tolerances (written here, used by every parity test):
  * integer add/min/max, float min/max, select (values and count): bit-exact;
  * f32 add: |gpu - p64| <= 1e-5 * sum_{j<=i} |x_j| + 1e-6, per element, where
    p64 is the oracle's fp64 prefix;
  * bf16/f16 add: |gpu - RN_T(p64)| <= ulp_T(RN_T(p64)) + 1e-5 * sum_{j<=i}|x_j|
    + 1e-6, with RN_T the oracle's round-to-nearest-even to the output type
    and ulp_T the spacing of T at that value (subnormal spacing near 0);
  * inputs whose every partial sum is exact in f32 (dyadic k/256 values):
    bit-exact for all three storage types;
  * row products: every grouping of the k <= i+1 factors of out[i] has at
    most k f32 roundings of relative size <= 2^-24 (no underflow on the
    inputs used), so |gpu - p64| <= ((1 + 2^-24)^(i+1) - 1) |p64|, plus
    ulp_T(RN_T(p64)) for bf16/f16 storage;
  * row min/max: bit-exact (the results are input values);
  * f64 add (1-D): |gpu - p| <= 1e-12 * sum_{j<=i} |x_j| + 1e-15, p the oracle's
    long-double prefix; u32/u64 and f64 min/max: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL, ABS = 1e-5, 1e-6
REL64, ABS64 = 1e-12, 1e-15  # f64 add: the f32 rule with f64's spacing


_BITS = {"i32": np.uint32, "f32": np.uint32, "u32": np.uint32, "i64": np.uint64, "u64": np.uint64,
         "f64": np.uint64}


def _np_cpu(t: torch.Tensor) -> np.ndarray:
    """A device tensor as a numpy array (unsigned 32/64-bit tensors through
    their signed bit patterns, which numpy then reads as unsigned)."""
    t = t.detach()
    if t.dtype == torch.uint32:
        return t.view(torch.int32).to("cpu").contiguous().numpy().view(np.uint32)
    if t.dtype == torch.uint64:
        return t.view(torch.int64).to("cpu").contiguous().numpy().view(np.uint64)
    return t.to("cpu").contiguous().numpy()


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_rows_close(gpu_out: torch.Tensor, x_cpu: torch.Tensor, dtype: str, inclusive: bool,
                      exact: bool = False):
    """Full comparison of a row scan with the oracle."""
    ref, p64, mag = oracle.scan_rows(x_cpu, dtype, inclusive, want_f64=True)
    if dtype == "f32":
        got = gpu_out.detach().to("cpu").numpy()
        if exact:
            bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))
            assert bad[0].size == 0, _report(bad, got, ref)
            return
        err = np.abs(got.astype(np.float64) - p64)
        bound = REL * mag + ABS
    else:
        gbits = bits16(gpu_out)
        if exact:
            bad = np.nonzero(gbits != ref)
            assert bad[0].size == 0, _report(bad, gbits, ref)
            return
        got = oracle.decode_half(gbits, dtype)
        want = oracle.decode_half(ref, dtype)
        err = np.abs(got - want)
        bound = oracle.ulp_array(want, dtype) + REL * mag + ABS
    bad = np.nonzero(~(err <= bound))
    if bad[0].size:
        i = tuple(b[0] for b in bad)
        raise AssertionError(f"{bad[0].size} elements out of tolerance; first at {i}: "
                             f"err {err[i]} bound {bound[i]}")


def assert_scan_matches(gpu_out: torch.Tensor, arr_cpu: torch.Tensor, n: int, dtype: str, op: str,
                        inclusive: bool = False):
    """1-D exclusive (or inclusive) scan of arr[0:n]: bit-exact except f32 add
    (tolerance)."""
    scan = oracle.inclusive_scan if inclusive else oracle.exclusive_scan
    got = _np_cpu(gpu_out[:n])
    if dtype in ("f32", "f64") and op == "add":
        _, p64, mag = scan(arr_cpu, n, dtype, op, want_f64=True)
        err = np.abs(got.astype(np.float64) - p64)
        bound = (REL * mag + ABS) if dtype == "f32" else (REL64 * mag + ABS64)
        bad = np.nonzero(~(err <= bound))[0]
        assert bad.size == 0, f"{bad.size} out of tolerance; first {bad[0]}: {got[bad[0]]} vs {p64[bad[0]]}"
        return
    ref = scan(arr_cpu, n, dtype, op)
    w = _BITS[dtype]
    bad = np.nonzero(got.view(w) != ref.view(w))[0]
    assert bad.size == 0, f"{bad.size} mismatches; first at {bad[0]}: {got[bad[0]]} vs {ref[bad[0]]}"


def assert_rows_op_close(gpu_out: torch.Tensor, x_cpu: torch.Tensor, dtype: str, op: str,
                         inclusive: bool):
    """Row scan with op in add / mul / min / max against the oracle."""
    if op == "add":
        assert_rows_close(gpu_out, x_cpu, dtype, inclusive)
        return
    ref, p64 = oracle.scan_rows_op(x_cpu, dtype, op, inclusive, want_f64=True)
    if op in ("min", "max"):
        got = (gpu_out.detach().to("cpu").numpy().view(np.uint32) if dtype == "f32"
               else bits16(gpu_out))
        want = ref.view(np.uint32) if dtype == "f32" else ref
        bad = np.nonzero(got != want)
        assert bad[0].size == 0, _report(bad, got, want)
        return
    k = np.arange(1, p64.shape[1] + 1, dtype=np.float64)[None, :]
    rel = np.expm1(k * np.log1p(2.0 ** -24))
    bound = rel * np.abs(p64)
    if dtype == "f32":
        got = gpu_out.detach().to("cpu").numpy().astype(np.float64)
        err = np.abs(got - p64)
    else:
        got = oracle.decode_half(bits16(gpu_out), dtype)
        want = oracle.decode_half(ref, dtype)
        err = np.abs(got - p64)
        bound = bound + oracle.ulp_array(want, dtype)
    bad = np.nonzero(~(err <= bound))
    if bad[0].size:
        i = tuple(b[0] for b in bad)
        raise AssertionError(f"{bad[0].size} elements out of tolerance; first at {i}: "
                             f"got {got[i]} p64 {p64[i]} err {err[i]} bound {bound[i]}")


def assert_reduce_matches(gpu_out: torch.Tensor, arr_cpu: torch.Tensor, n: int, dtype: str, op: str):
    """out[0] of a reduction: bit-exact except f32 add, which must lie within
    REL * sum|x| + ABS of the fp64 sum."""
    got = _np_cpu(gpu_out[:1])[0]
    if dtype in ("f32", "f64") and op == "add":
        _, s64, m64 = oracle.reduce(arr_cpu, n, dtype, op, want_f64=True)
        rel, ab = (REL, ABS) if dtype == "f32" else (REL64, ABS64)
        assert abs(float(got) - s64) <= rel * m64 + ab, f"{got} vs {s64} (sum|x| {m64})"
        return
    ref = oracle.reduce(arr_cpu, n, dtype, op)
    w = _BITS[dtype]
    assert np.array([got]).view(w)[0] == np.array([ref]).view(w)[0], f"{got} vs {ref}"


def assert_select_matches(gpu_out: torch.Tensor, gpu_num: torch.Tensor, arr_cpu, flags_cpu, n: int):
    ref, k = oracle.select(arr_cpu, flags_cpu, n)
    got_k = int(gpu_num.item())
    assert got_k == k, f"num_out {got_k} != {k}"
    got = gpu_out[:k].detach().to("cpu").contiguous().view(torch.int32).numpy().view(np.uint32)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches; first at {bad[0]}"


def _report(bad, got, ref):
    i = tuple(b[0] for b in bad)
    return f"{bad[0].size} mismatches; first at {i}: {got[i]} vs {ref[i]}"
