"""All-core CPU scans (``cpu_allcore.c``, pthreads): the row scan and the
1-D exclusive scan -- a MEASUREMENT BASELINE for ``bench.py``'s CPU leg only.
It is not the oracle (the oracle stays single-threaded and fp64) and the GPU
product never imports it."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cpu_allcore.c")
_LIB = os.path.join(_HERE, "libcpuallcore.so")
_DT = {"f32": 0, "bf16": 1, "f16": 2, "i32": 3, "i64": 4}
_OP = {"add": 0, "min": 1, "max": 2}
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.cpu_allcore_scan_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int]
        L.cpu_allcore_scan_rows.restype = ctypes.c_int
        L.cpu_allcore_exclusive_scan.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int]
        L.cpu_allcore_exclusive_scan.restype = ctypes.c_int
        _lib = L
    return _lib


def cores() -> int:
    """Host cores this process may run on."""
    return len(os.sched_getaffinity(0))


def scan_rows(x, dtype: str, inclusive: bool, threads: int, out=None) -> np.ndarray:
    """Row scan of a contiguous 2-D array (f32 values, or bf16/f16 bit
    patterns as 16-bit integers); returns the output in the same form."""
    if hasattr(x, "numpy"):  # a CPU torch tensor (bf16/f16 viewed as 16-bit integers)
        x = x.contiguous()
        if dtype != "f32":
            import torch
            x = x.view(torch.int16)
        x = x.numpy()
    a = np.ascontiguousarray(x)
    if dtype != "f32":
        a = a.view(np.uint16)
    y = np.empty_like(a) if out is None else out
    rows, n = a.shape
    rc = _get().cpu_allcore_scan_rows(a.ctypes.data, y.ctypes.data, rows, n, _DT[dtype], int(bool(inclusive)),
                                      threads)
    if rc != 0:
        raise RuntimeError("cpu_allcore_scan_rows failed")
    return y


def exclusive_scan(x, n: int, dtype: str, op: str, threads: int, out=None) -> np.ndarray:
    """Exclusive scan of the first n elements of a 1-D i32/i64/f32 array (a
    CPU torch tensor or numpy array); returns out (the first n written)."""
    if hasattr(x, "numpy"):
        x = x.numpy()
    a = np.ascontiguousarray(x)
    if a.ndim != 1 or n < 0 or n > a.shape[0]:
        raise ValueError("exclusive_scan: a 1-D array with at least n elements")
    y = np.empty_like(a) if out is None else out
    rc = _get().cpu_allcore_exclusive_scan(a.ctypes.data, y.ctypes.data, n, _DT[dtype], _OP[op], threads)
    if rc != 0:
        raise RuntimeError("cpu_allcore_exclusive_scan failed")
    return y
