"""CPU oracle for the prefix-scan library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The product
package never imports it, and this package imports nothing from the product.

It wraps ``mt_oracle.c`` (plain, single-threaded C; fp64 accumulation for
floats) through ctypes and works on numpy arrays / CPU torch tensors. See the
C file's header for the passages each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mt_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, F16, I32, I64, U32, U64, F64 = 0, 1, 2, 3, 4, 5, 6, 7
ADD, MIN, MAX, MUL = 0, 1, 2, 3
DTYPES = {"f32": F32, "bf16": BF16, "f16": F16, "i32": I32, "i64": I64, "u32": U32, "u64": U64,
          "f64": F64}
OPS = {"add": ADD, "min": MIN, "max": MAX, "mul": MUL}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
            "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.oracle_scan_rows.argtypes = [p, p, p, p, i64, i64, i32, i32]
        L.oracle_scan_rows.restype = i32
        L.oracle_exclusive_scan.argtypes = [p, p, p, p, i64, i32, i32]
        L.oracle_exclusive_scan.restype = i32
        L.oracle_scan_rows_op.argtypes = [p, p, p, i64, i64, i32, i32, i32]
        L.oracle_scan_rows_op.restype = i32
        L.oracle_inclusive_scan.argtypes = [p, p, p, p, i64, i32, i32]
        L.oracle_inclusive_scan.restype = i32
        L.oracle_reduce.argtypes = [p, p, p, p, i64, i32, i32]
        L.oracle_reduce.restype = i32
        L.oracle_select.argtypes = [p, p, p, i64]
        L.oracle_select.restype = i64
        L.oracle_select_wide.argtypes = [p, p, p, i64, i32]
        L.oracle_select_wide.restype = i64
        L.oracle_reduce_by_key_add.argtypes = [p, p, p, p, p, p, i64, i32, i32]
        L.oracle_reduce_by_key_add.restype = i64
        L.oracle_decode_half.argtypes = [p, p, i64, i32]
        L.oracle_decode_half.restype = None
        L.oracle_encode_half.argtypes = [p, p, i64, i32]
        L.oracle_encode_half.restype = None
        L.oracle_ulp.argtypes = [ctypes.c_double, i32]
        L.oracle_ulp.restype = ctypes.c_double
        _lib = L
    return _lib


def _np(x) -> np.ndarray:
    """A C-contiguous numpy view of a CPU tensor or array (bf16/f16 as u16 bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype in (torch.bfloat16, torch.float16):
                x = x.view(torch.int16)
            elif x.dtype == torch.uint32:  # numpy reads the signed bits back as unsigned
                return np.ascontiguousarray(x.view(torch.int32).numpy()).view(np.uint32)
            elif x.dtype == torch.uint64:
                return np.ascontiguousarray(x.view(torch.int64).numpy()).view(np.uint64)
            return np.ascontiguousarray(x.numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


_STORE_NP = {F32: np.float32, BF16: np.uint16, F16: np.uint16}


def scan_rows(x, dtype: str, inclusive: bool, want_f64: bool = False):
    """Row-wise sum scan of a [rows, n] input.

    Returns the output in storage form (f32 array, or u16 bit patterns for
    bf16/f16); with ``want_f64`` also returns (prefix64, abs64).
    """
    d = DTYPES[dtype]
    a = _np(x)
    rows, n = a.shape
    out = np.empty((rows, n), dtype=_STORE_NP[d])
    p64 = np.empty((rows, n), dtype=np.float64) if want_f64 else None
    m64 = np.empty((rows, n), dtype=np.float64) if want_f64 else None
    rc = lib().oracle_scan_rows(_ptr(a), _ptr(out), _ptr(p64) if want_f64 else None,
                                _ptr(m64) if want_f64 else None, rows, n, d, int(bool(inclusive)))
    if rc != 0:
        raise ValueError("oracle_scan_rows rejected its arguments")
    return (out, p64, m64) if want_f64 else out


def scan_rows_op(x, dtype: str, op: str, inclusive: bool, want_f64: bool = False):
    """Row-wise scan of a [rows, n] input with op in add / mul / min / max.

    Returns the output in storage form (f32 array, or u16 bit patterns for
    bf16/f16); with ``want_f64`` also the fp64 prefix.
    """
    d, o = DTYPES[dtype], OPS[op]
    a = _np(x)
    rows, n = a.shape
    out = np.empty((rows, n), dtype=_STORE_NP[d])
    p64 = np.empty((rows, n), dtype=np.float64) if want_f64 else None
    rc = lib().oracle_scan_rows_op(_ptr(a), _ptr(out), _ptr(p64) if want_f64 else None, rows, n, d,
                                   o, int(bool(inclusive)))
    if rc != 0:
        raise ValueError("oracle_scan_rows_op rejected its arguments")
    return (out, p64) if want_f64 else out


_SCAN_NP = {F32: np.float32, I32: np.int32, I64: np.int64, U32: np.uint32, U64: np.uint64,
            F64: np.float64}


def exclusive_scan(arr, n: int, dtype: str, op: str, want_f64: bool = False):
    """Exclusive scan of arr[0:n]; returns out[0:n] (and prefix64/abs64 for
    f32 add when ``want_f64``)."""
    d, o = DTYPES[dtype], OPS[op]
    a = _np(arr)[:n]
    a = np.ascontiguousarray(a)
    out = np.empty((n,), dtype=_SCAN_NP[d])
    f64 = want_f64 and d in (F32, F64) and o == ADD
    p64 = np.empty((n,), dtype=np.float64) if f64 else None
    m64 = np.empty((n,), dtype=np.float64) if f64 else None
    rc = lib().oracle_exclusive_scan(_ptr(a), _ptr(out), _ptr(p64) if f64 else None,
                                     _ptr(m64) if f64 else None, n, d, o)
    if rc != 0:
        raise ValueError("oracle_exclusive_scan rejected its arguments")
    return (out, p64, m64) if f64 else out


def inclusive_scan(arr, n: int, dtype: str, op: str, want_f64: bool = False):
    """Inclusive scan of arr[0:n]: out[i] = op(arr[0..=i]); returns out[0:n]
    (and prefix64/abs64 for f32 add when ``want_f64``)."""
    d, o = DTYPES[dtype], OPS[op]
    a = np.ascontiguousarray(_np(arr)[:n])
    out = np.empty((n,), dtype=_SCAN_NP[d])
    f64 = want_f64 and d in (F32, F64) and o == ADD
    p64 = np.empty((n,), dtype=np.float64) if f64 else None
    m64 = np.empty((n,), dtype=np.float64) if f64 else None
    rc = lib().oracle_inclusive_scan(_ptr(a), _ptr(out), _ptr(p64) if f64 else None,
                                     _ptr(m64) if f64 else None, n, d, o)
    if rc != 0:
        raise ValueError("oracle_inclusive_scan rejected its arguments")
    return (out, p64, m64) if f64 else out


def reduce(arr, n: int, dtype: str, op: str, want_f64: bool = False):
    """op(arr[0:n]) as a numpy scalar of the dtype (the identity for n == 0);
    with ``want_f64`` for f32 add also the fp64 sum and the sum of |x|."""
    d, o = DTYPES[dtype], OPS[op]
    a = np.ascontiguousarray(_np(arr)[:n])
    if a.size == 0:
        a = np.zeros((1,), dtype=_SCAN_NP[d])
    out = np.empty((1,), dtype=_SCAN_NP[d])
    s64 = np.zeros((1,), dtype=np.float64)
    m64 = np.zeros((1,), dtype=np.float64)
    rc = lib().oracle_reduce(_ptr(a), _ptr(out), _ptr(s64), _ptr(m64), n, d, o)
    if rc != 0:
        raise ValueError("oracle_reduce rejected its arguments")
    f64 = want_f64 and d in (F32, F64) and o == ADD
    return (out[0], float(s64[0]), float(m64[0])) if f64 else out[0]


def select(arr, flags, n: int):
    """Stream compaction of 4-byte elements; returns (out[0:num_out] as u32
    bit patterns, num_out)."""
    a = np.ascontiguousarray(_np(arr)[:n]).view(np.uint32)
    f = np.ascontiguousarray(_np(flags)[:n]).view(np.uint8)
    out = np.empty((max(n, 1),), dtype=np.uint32)
    k = lib().oracle_select(_ptr(a), _ptr(f), _ptr(out), n)
    return out[:k].copy(), int(k)


def select_wide(arr, flags, n: int, elem_bytes: int):
    """Stream compaction of elements of elem_bytes bytes; returns
    (out[0:num_out], num_out). out holds u32 / u64 bit patterns for 4- / 8-byte
    elements, else a [num_out, elem_bytes] uint8 array (one struct per row).
    arr is any array whose first n * elem_bytes bytes are the n elements."""
    f = np.ascontiguousarray(_np(flags)[:n]).view(np.uint8)
    if elem_bytes in (4, 8):
        w = np.uint32 if elem_bytes == 4 else np.uint64
        a = np.ascontiguousarray(_np(arr)[:n]).view(w)
        out = np.empty((max(n, 1),), dtype=w)
    else:
        a = np.ascontiguousarray(_np(arr)).reshape(-1).view(np.uint8)[:n * elem_bytes]
        if a.size != n * elem_bytes:
            raise ValueError("arr holds fewer than n elements")
        out = np.empty((max(n, 1), max(elem_bytes, 1)), dtype=np.uint8)
    k = lib().oracle_select_wide(_ptr(a), _ptr(f), _ptr(out), n, elem_bytes)
    if k < 0:
        raise ValueError("oracle_select_wide rejected its arguments")
    return out[:k].copy(), int(k)


def decode_half(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_decode_half(_ptr(b), _ptr(out), b.size, DTYPES[dtype])
    return out


def encode_half(x: np.ndarray, dtype: str) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().oracle_encode_half(_ptr(a), _ptr(out), a.size, DTYPES[dtype])
    return out


def ulp(v: float, dtype: str) -> float:
    return lib().oracle_ulp(float(v), DTYPES[dtype])


def ulp_array(v: np.ndarray, dtype: str) -> np.ndarray:
    """Element-wise spacing of the output format at |v| (numpy, vectorised
    form of ``ulp``; the C function pins it in the tests)."""
    frac_bits, emin = {"f32": (23, -126), "bf16": (7, -126), "f16": (10, -14)}[dtype]
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e2 = np.frexp(a)
    E = np.where(a == 0.0, emin, np.maximum(e2 - 1, emin))
    return np.ldexp(1.0, (E - frac_bits).astype(np.int32))


_RBK_NP = {I32: np.int32, U32: np.uint32, F32: np.float32}


def reduce_by_key_add(keys, vals, n: int, key_dtype: str, val_dtype: str, want_f64: bool = False):
    """Runs of consecutive equal keys -> (keys_out[0:r], values_out[0:r], r);
    with ``want_f64`` for f32 values also each run's fp64 sum and sum of |v|."""
    kd, vd = DTYPES[key_dtype], DTYPES[val_dtype]
    k = np.ascontiguousarray(_np(keys)[:n])
    v = np.ascontiguousarray(_np(vals)[:n])
    ko = np.empty((max(n, 1),), dtype=_RBK_NP[kd])
    vo = np.empty((max(n, 1),), dtype=_RBK_NP[vd])
    s64 = np.empty((max(n, 1),), dtype=np.float64)
    m64 = np.empty((max(n, 1),), dtype=np.float64)
    r = lib().oracle_reduce_by_key_add(_ptr(k), _ptr(v), _ptr(ko), _ptr(vo), _ptr(s64), _ptr(m64), n,
                                       kd, vd)
    if r < 0:
        raise ValueError("oracle_reduce_by_key_add rejected its arguments")
    if want_f64:
        return ko[:r].copy(), vo[:r].copy(), int(r), s64[:r].copy(), m64[:r].copy()
    return ko[:r].copy(), vo[:r].copy(), int(r)

