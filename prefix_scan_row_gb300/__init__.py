"""Python binding of libmtscan.so (include/mt_scan.h): prefix scans on one
NVIDIA GB300.

The functions here only marshal arguments (pointers, sizes, the current CUDA
stream) into the C ABI; every step of the scan runs in the library's CUDA
kernels. There is no fallback: if the shared library is missing or fails to
load, importing this package raises.

Names and arguments follow the C ABI:

* ``mt_scan_rows(inp, out, inclusive)`` -- row-wise sum scan of a contiguous
  [rows, n] f32/bf16/f16 CUDA tensor.
* ``mt_scan_rows_op(inp, out, op, inclusive)`` -- the same with op in
  add / mul / max / min.
* ``mt_exclusive_scan(arr, out, scratch, n_dev, op)`` -- device-wide exclusive
  add/min/max over i32/i64/f32 with the live count in a device int32.
* ``mt_inclusive_scan(arr, out, scratch, n_dev, op)`` -- the inclusive form
  (in place allowed).
* ``mt_reduce(arr, out, scratch, n_dev, op)`` -- out[0] = op(arr[0:n]).
* ``mt_select(arr, flags, out, num_out, scratch, n_dev)`` -- stream compaction
  (``mt_select_wide`` for 8-byte elements).
* ``mt_reduce_by_key_add(keys_in, values_in, keys_out, values_out, num_runs,
  scratch, n_dev)`` -- run-length sums of consecutive equal keys.
* ``mt_scan_scratch_slots(capacity, dtype, kind)`` -- scratch sizing.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmtscan.so")
LIB_CHECKED_PATH = os.path.join(_HERE, "libmtscan_checked.so")  # the bounds-checked build

MT_F32, MT_BF16, MT_F16, MT_I32, MT_I64, MT_U32, MT_U64, MT_F64 = 0, 1, 2, 3, 4, 5, 6, 7
MT_ADD, MT_MIN, MT_MAX, MT_MUL = 0, 1, 2, 3
MT_SCRATCH_SCAN, MT_SCRATCH_SELECT, MT_SCRATCH_REDUCE, MT_SCRATCH_REDUCE_BY_KEY = 1, 2, 3, 4
MT_OK = 0
MT_ERR_ARG, MT_ERR_DTYPE, MT_ERR_ALIAS, MT_ERR_CUDA, MT_ERR_LOOKBACK_TIMEOUT, MT_ERR_ALIGN = (
    -1, -2, -3, -4, -5, -6)
MT_ERR_TOO_LARGE = -7
MT_ERR_MEMORY = -8
MT_ERR_BOUNDS = -9
MT_NOALLOC_SCRATCH_BYTES = 1 << 20

DTYPE_CODE = {torch.float32: MT_F32, torch.bfloat16: MT_BF16, torch.float16: MT_F16,
              torch.int32: MT_I32, torch.int64: MT_I64, torch.uint32: MT_U32, torch.uint64: MT_U64,
              torch.float64: MT_F64}
OP_CODE = {"add": MT_ADD, "min": MT_MIN, "max": MT_MAX, "mul": MT_MUL}

EXPORTS = ("mt_scan_rows", "mt_scan_rows_op", "mt_exclusive_scan", "mt_inclusive_scan", "mt_reduce", "mt_select",
           "mt_select_wide", "mt_reduce_by_key_add", "mt_scan_scratch_slots",
           "mt_scan_status", "mt_scan_launches", "mt_scan_strerror", "mt_scan_debug_lookback",
           "mt_scan_rows_noalloc", "mt_scan_rows_scratch_slots", "mt_scan_build_checked")


class ScanError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mt_scan_strerror(code)} ({code})")


def _load(path: str):
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`"
            " (the scan library has no CPU fallback)")
    L = ctypes.CDLL(path)
    p, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
    L.mt_scan_rows.argtypes = [p, p, i64, i64, i32, i32, p]
    L.mt_scan_rows.restype = i32
    L.mt_scan_rows_op.argtypes = [p, p, i64, i64, i32, i32, i32, p]
    L.mt_scan_rows_op.restype = i32
    L.mt_exclusive_scan.argtypes = [p, p, p, p, i32, i32, p]
    L.mt_exclusive_scan.restype = i32
    L.mt_inclusive_scan.argtypes = [p, p, p, p, i32, i32, p]
    L.mt_inclusive_scan.restype = i32
    L.mt_reduce.argtypes = [p, p, p, p, i32, i32, p]
    L.mt_reduce.restype = i32
    L.mt_select.argtypes = [p, p, p, p, p, p, p]
    L.mt_select_wide.argtypes = [p, p, p, p, p, p, i32, p]
    L.mt_select_wide.restype = i32
    L.mt_reduce_by_key_add.argtypes = [p, p, p, p, p, p, p, i32, i32, p]
    L.mt_reduce_by_key_add.restype = i32
    L.mt_select.restype = i32
    L.mt_scan_scratch_slots.argtypes = [i64, i32, i32]
    L.mt_scan_scratch_slots.restype = i64
    L.mt_scan_status.argtypes = [p]
    L.mt_scan_status.restype = i32
    L.mt_scan_launches.argtypes = []
    L.mt_scan_launches.restype = ctypes.c_uint64
    L.mt_scan_strerror.argtypes = [i32]
    L.mt_scan_strerror.restype = ctypes.c_char_p
    L.mt_scan_debug_lookback.argtypes = [i64, u32]
    L.mt_scan_debug_lookback.restype = i32
    L.mt_scan_rows_noalloc.argtypes = [p, p, i64, i64, i32, i32, p]
    L.mt_scan_rows_noalloc.restype = i32
    L.mt_scan_rows_scratch_slots.argtypes = [i64, i64, i32]
    L.mt_scan_rows_scratch_slots.restype = i64
    L.mt_scan_build_checked.argtypes = []
    L.mt_scan_build_checked.restype = i32
    return L


def _check(code: int, where: str) -> None:
    if code != MT_OK:
        raise ScanError(code, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    return 0 if t is None else (t if isinstance(t, int) else t.data_ptr())


def _contiguous(**tensors) -> None:
    """The library sees flat memory: a strided view would be read as such."""
    for name, t in tensors.items():
        if isinstance(t, torch.Tensor) and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


class Library:
    """The calls of one loaded build of the C ABI: the ordinary library, or
    (load_checked) its bounds-checked twin. Each method marshals torch
    tensors into the C call of the same name."""

    def __init__(self, path: str):
        self.path = path
        self.lib = _load(path)

    def mt_scan_strerror(self, code: int) -> str:
        return self.lib.mt_scan_strerror(int(code)).decode()

    def mt_scan_rows(self, inp: torch.Tensor, out: torch.Tensor, inclusive: bool, stream=None) -> None:
        """Row-wise sum scan of a contiguous 2-D (or 1-D = one row) CUDA tensor."""
        if inp.dim() == 1:
            rows, n = 1, inp.shape[0]
        else:
            rows, n = inp.shape
        if out.shape != inp.shape or out.dtype != inp.dtype:
            raise ValueError("out must match inp in shape and dtype")
        if not (inp.is_contiguous() and out.is_contiguous()):
            raise ValueError("inp and out must be contiguous")
        code = DTYPE_CODE.get(inp.dtype, -99)
        _check(self.lib.mt_scan_rows(_ptr(inp), _ptr(out), rows, n, code, int(bool(inclusive)),
                                     _stream(stream)), "mt_scan_rows")

    def mt_scan_rows_op(self, inp: torch.Tensor, out: torch.Tensor, op: str, inclusive: bool,
                        stream=None) -> None:
        """Row-wise scan with op in 'add' | 'mul' | 'max' | 'min'."""
        if inp.dim() == 1:
            rows, n = 1, inp.shape[0]
        else:
            rows, n = inp.shape
        if out.shape != inp.shape or out.dtype != inp.dtype:
            raise ValueError("out must match inp in shape and dtype")
        if not (inp.is_contiguous() and out.is_contiguous()):
            raise ValueError("inp and out must be contiguous")
        code = DTYPE_CODE.get(inp.dtype, -99)
        _check(self.lib.mt_scan_rows_op(_ptr(inp), _ptr(out), rows, n, code, OP_CODE[op],
                                        int(bool(inclusive)), _stream(stream)), "mt_scan_rows_op")

    def mt_exclusive_scan(self, arr: torch.Tensor, out: torch.Tensor, scratch: torch.Tensor,
                          n_dev: torch.Tensor, op: str, stream=None) -> None:
        """Exclusive scan of arr[0:*n_dev] into out (op: 'add' | 'min' | 'max')."""
        if out.dtype != arr.dtype:
            raise ValueError("out must have arr's dtype")
        if n_dev.dtype != torch.int32:
            raise ValueError("n_dev must be an int32 device tensor")
        _contiguous(arr=arr, out=out, scratch=scratch)
        code = DTYPE_CODE.get(arr.dtype, -99)
        _check(self.lib.mt_exclusive_scan(_ptr(arr), _ptr(out), _ptr(scratch), _ptr(n_dev), code,
                                          OP_CODE[op], _stream(stream)), "mt_exclusive_scan")

    def mt_inclusive_scan(self, arr: torch.Tensor, out: torch.Tensor, scratch: torch.Tensor,
                          n_dev: torch.Tensor, op: str, stream=None) -> None:
        """Inclusive scan of arr[0:*n_dev] into out (out may be arr)."""
        if out.dtype != arr.dtype:
            raise ValueError("out must have arr's dtype")
        if n_dev.dtype != torch.int32:
            raise ValueError("n_dev must be an int32 device tensor")
        _contiguous(arr=arr, out=out, scratch=scratch)
        code = DTYPE_CODE.get(arr.dtype, -99)
        _check(self.lib.mt_inclusive_scan(_ptr(arr), _ptr(out), _ptr(scratch), _ptr(n_dev), code,
                                          OP_CODE[op], _stream(stream)), "mt_inclusive_scan")

    def mt_reduce(self, arr: torch.Tensor, out: torch.Tensor, scratch: torch.Tensor, n_dev: torch.Tensor,
                  op: str, stream=None) -> None:
        """out[0] = op(arr[0:*n_dev]) (the identity for an empty input)."""
        if out.dtype != arr.dtype:
            raise ValueError("out must have arr's dtype")
        if n_dev.dtype != torch.int32:
            raise ValueError("n_dev must be an int32 device tensor")
        _contiguous(arr=arr, scratch=scratch)
        code = DTYPE_CODE.get(arr.dtype, -99)
        _check(self.lib.mt_reduce(_ptr(arr), _ptr(out), _ptr(scratch), _ptr(n_dev), code, OP_CODE[op],
                                  _stream(stream)), "mt_reduce")

    def mt_select(self, arr: torch.Tensor, flags: torch.Tensor, out: torch.Tensor, num_out: torch.Tensor,
                  scratch: torch.Tensor, n_dev: torch.Tensor, stream=None) -> None:
        """Stream compaction of 4-byte elements by exactly-0/1 uint8 flags."""
        if arr.element_size() != 4 or out.element_size() != 4:
            raise ValueError("select copies 4-byte elements")
        if flags.dtype != torch.uint8 or num_out.dtype != torch.int32 or n_dev.dtype != torch.int32:
            raise ValueError("flags must be uint8, num_out and n_dev int32")
        _contiguous(arr=arr, flags=flags, out=out, scratch=scratch)
        _check(self.lib.mt_select(_ptr(arr), _ptr(flags), _ptr(out), _ptr(num_out), _ptr(scratch),
                                  _ptr(n_dev), _stream(stream)), "mt_select")

    def mt_select_wide(self, arr: torch.Tensor, flags: torch.Tensor, out: torch.Tensor, num_out: torch.Tensor,
                       scratch: torch.Tensor, n_dev: torch.Tensor, stream=None) -> None:
        """Stream compaction of 4- or 8-byte elements, or of structs: a 1-D arr
        holds one element per entry, an [n, ...] arr one struct per row (its
        trailing dimensions), copied bit for bit."""
        eb = arr.element_size() * math.prod(arr.shape[1:])
        if out.element_size() * math.prod(out.shape[1:]) != eb:
            raise ValueError("out's elements must have arr's size")
        if flags.dtype != torch.uint8 or num_out.dtype != torch.int32 or n_dev.dtype != torch.int32:
            raise ValueError("flags must be uint8, num_out and n_dev int32")
        _contiguous(arr=arr, flags=flags, out=out, scratch=scratch)
        _check(self.lib.mt_select_wide(_ptr(arr), _ptr(flags), _ptr(out), _ptr(num_out), _ptr(scratch),
                                       _ptr(n_dev), eb, _stream(stream)), "mt_select_wide")

    def mt_reduce_by_key_add(self, keys_in: torch.Tensor, values_in: torch.Tensor, keys_out: torch.Tensor,
                             values_out: torch.Tensor, num_runs: torch.Tensor, scratch: torch.Tensor,
                             n_dev: torch.Tensor, stream=None) -> None:
        """Runs of consecutive equal keys -> (key, sum of values); i32/u32/f32."""
        if keys_out.dtype != keys_in.dtype or values_out.dtype != values_in.dtype:
            raise ValueError("outputs must have their inputs' dtypes")
        if num_runs.dtype != torch.int32 or n_dev.dtype != torch.int32:
            raise ValueError("num_runs and n_dev must be int32")
        _contiguous(keys_in=keys_in, values_in=values_in, keys_out=keys_out, values_out=values_out,
                    scratch=scratch)
        _check(self.lib.mt_reduce_by_key_add(_ptr(keys_in), _ptr(values_in), _ptr(keys_out), _ptr(values_out),
                                             _ptr(num_runs), _ptr(scratch), _ptr(n_dev),
                                             DTYPE_CODE.get(keys_in.dtype, -99), DTYPE_CODE.get(values_in.dtype, -99),
                                             _stream(stream)), "mt_reduce_by_key_add")

    def mt_scan_scratch_slots(self, capacity: int, dtype, kind: int) -> int:
        code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
        r = self.lib.mt_scan_scratch_slots(int(capacity), code, int(kind))
        if r < 0:
            raise ValueError("mt_scan_scratch_slots: bad capacity, dtype or kind")
        return r

    def mt_scan_rows_scratch_slots(self, rows: int, n: int, dtype) -> int:
        """8-byte slots of look-back workspace a [rows, n] row scan of `dtype`
        takes (from the library's pool, or from mt_scan_rows_noalloc's array);
        0 when every row fits in one tile."""
        code = DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
        r = self.lib.mt_scan_rows_scratch_slots(int(rows), int(n), code)
        if r < 0:
            raise ValueError("mt_scan_rows_scratch_slots: bad size or dtype")
        return r

    def alloc_scratch(self, capacity: int, dtype, kind: int, device="cuda") -> torch.Tensor:
        """Caller-owned scratch of mt_scan_scratch_slots(...) 8-byte slots."""
        return torch.empty(self.mt_scan_scratch_slots(capacity, dtype, kind), dtype=torch.int64,
                           device=device)

    def mt_scan_status(self, stream=None) -> int:
        """Synchronise the stream, then read and clear the device error words."""
        return self.lib.mt_scan_status(_stream(stream))

    def mt_scan_launches(self) -> int:
        return self.lib.mt_scan_launches()

    def mt_scan_build_checked(self) -> bool:
        return bool(self.lib.mt_scan_build_checked())

    def mt_scan_debug_lookback(self, skip_publish_tile: int = -1, spin_limit: int = 0) -> None:
        self.lib.mt_scan_debug_lookback(int(skip_publish_tile), int(spin_limit))

    def mt_scan_rows_noalloc(self, inp: torch.Tensor, out: torch.Tensor, inclusive: bool, stream=None) -> None:
        """mt_scan_rows without any device allocation, for callers that may not
        allocate: the look-back records of long rows live in a fixed 1 MiB array
        inside the library. Raises ScanError(MT_ERR_TOO_LARGE) for a shape that
        needs more (mt_scan_rows_scratch_slots(rows, n, dtype) * 8 above
        MT_NOALLOC_SCRATCH_BYTES). The first long-row call in a CUDA context
        looks up that array's address there; calls that overlap on the GPU must
        not be made."""
        if inp.dim() == 1:
            rows, n = 1, inp.shape[0]
        else:
            rows, n = inp.shape
        if out.shape != inp.shape or out.dtype != inp.dtype:
            raise ValueError("out must match inp in shape and dtype")
        if not (inp.is_contiguous() and out.is_contiguous()):
            raise ValueError("inp and out must be contiguous")
        code = DTYPE_CODE.get(inp.dtype, -99)
        _check(self.lib.mt_scan_rows_noalloc(_ptr(inp), _ptr(out), rows, n, code, int(bool(inclusive)),
                                             _stream(stream)), "mt_scan_rows_noalloc")


_default = Library(LIB_PATH)
lib = _default.lib
mt_scan_strerror = _default.mt_scan_strerror
mt_scan_rows = _default.mt_scan_rows
mt_scan_rows_op = _default.mt_scan_rows_op
mt_exclusive_scan = _default.mt_exclusive_scan
mt_inclusive_scan = _default.mt_inclusive_scan
mt_reduce = _default.mt_reduce
mt_select = _default.mt_select
mt_select_wide = _default.mt_select_wide
mt_reduce_by_key_add = _default.mt_reduce_by_key_add
mt_scan_scratch_slots = _default.mt_scan_scratch_slots
mt_scan_rows_scratch_slots = _default.mt_scan_rows_scratch_slots
alloc_scratch = _default.alloc_scratch
mt_scan_status = _default.mt_scan_status
mt_scan_launches = _default.mt_scan_launches
mt_scan_build_checked = _default.mt_scan_build_checked
mt_scan_debug_lookback = _default.mt_scan_debug_lookback
mt_scan_rows_noalloc = _default.mt_scan_rows_noalloc


def load_checked() -> Library:
    """The bounds-checked build (libmtscan_checked.so): the same calls, whose
    kernels check every store and shared-memory access against its buffer
    and report a bad one as MT_ERR_BOUNDS through mt_scan_status() instead of
    making it. For tests and debugging."""
    return Library(LIB_CHECKED_PATH)
