"""CPU checks of the C ABI: the library builds, loads, exports every function
include/mt_scan.h declares, and rejects bad arguments on the host before any
CUDA call. No kernel is launched here."""
import ctypes
import os
import re
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mt_scan.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    L = ctypes.CDLL(path)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mt_scan_rows.argtypes = [p, p, i64, i64, i32, i32, p]
    L.mt_scan_rows_op.argtypes = [p, p, i64, i64, i32, i32, i32, p]
    L.mt_exclusive_scan.argtypes = [p, p, p, p, i32, i32, p]
    L.mt_inclusive_scan.argtypes = [p, p, p, p, i32, i32, p]
    L.mt_reduce.argtypes = [p, p, p, p, i32, i32, p]
    L.mt_select.argtypes = [p, p, p, p, p, p, p]
    L.mt_select_wide.argtypes = [p, p, p, p, p, p, i32, p]
    L.mt_reduce_by_key_add.argtypes = [p, p, p, p, p, p, p, i32, i32, p]
    L.mt_scan_scratch_slots.argtypes = [i64, i32, i32]
    L.mt_scan_scratch_slots.restype = i64
    L.mt_scan_strerror.argtypes = [i32]
    L.mt_scan_strerror.restype = ctypes.c_char_p
    L.mt_scan_launches.restype = ctypes.c_uint64
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mt_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for name in names:
        assert hasattr(lib, name), f"{name} declared in mt_scan.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mt_\w+)", out))
    assert set(names) <= exported


def test_checked_build_exports_the_same_calls(lib):
    """The bounds-checked twin exports every declared call too, and says which
    build it is (no kernel is launched)."""
    import __graft_entry__
    checked = ctypes.CDLL(__graft_entry__._build_module().build(checked=True))
    out = subprocess.run(["nm", "-D", "--defined-only", checked._name], capture_output=True, text=True).stdout
    assert set(declared_functions()) <= set(re.findall(r"\bT (mt_\w+)", out))
    assert checked.mt_scan_build_checked() == 1
    assert lib.mt_scan_build_checked() == 0


def test_binding_names_match_header():
    import prefix_scan_row_gb300 as m
    assert sorted(m.EXPORTS) == declared_functions()
    for name in m.EXPORTS:
        assert callable(getattr(m, name))


F32, BF16, F16, I32, I64 = 0, 1, 2, 3, 4
OK, ARG, DTYPE, ALIAS, CUDA, TIMEOUT, ALIGN = 0, -1, -2, -3, -4, -5, -6
A, B, S, N = 0x10000, 0x20000, 0x30000, 0x40000  # fake, 16-byte aligned; never dereferenced


def test_rows_host_checks(lib):
    assert lib.mt_scan_rows(A, B, -1, 5, F32, 1, None) == ARG
    assert lib.mt_scan_rows(A, B, 5, -1, F32, 1, None) == ARG
    assert lib.mt_scan_rows(A, B, 2, 2, I32, 1, None) == DTYPE
    assert lib.mt_scan_rows(A, B, 2, 2, 9, 1, None) == DTYPE
    assert lib.mt_scan_rows(A, B, 0, 7, F32, 1, None) == OK       # empty: no-op
    assert lib.mt_scan_rows(None, None, 3, 0, BF16, 0, None) == OK  # empty: no-op
    assert lib.mt_scan_rows(None, B, 2, 2, F32, 1, None) == ARG
    assert lib.mt_scan_rows(A + 2, B, 2, 2, F32, 1, None) == ALIGN
    assert lib.mt_scan_rows(A + 1, B, 2, 2, F16, 1, None) == ALIGN
    assert lib.mt_scan_rows(A, B, 1 << 40, 1 << 40, F32, 1, None) == ARG  # size overflow


def test_rows_op_host_checks(lib):
    f = lib.mt_scan_rows_op
    assert f(A, B, 2, 8, F32, 4, 1, None) == ARG
    assert f(A, B, 2, 8, F32, -1, 1, None) == ARG
    assert f(A, B, -1, 8, F32, 3, 1, None) == ARG
    assert f(A, B, 2, 8, I32, 3, 1, None) == DTYPE
    assert f(A, B, 0, 8, F32, 3, 1, None) == 0  # empty
    assert f(A + 2, B, 2, 8, F32, 3, 1, None) == ALIGN
    # the 1-D calls take add / min / max only
    assert lib.mt_exclusive_scan(A, B, S, N, F32, 3, None) == ARG


def test_exclusive_scan_host_checks(lib):
    assert lib.mt_exclusive_scan(A, B, S, N, BF16, 0, None) == DTYPE
    assert lib.mt_exclusive_scan(A, B, S, N, I32, 3, None) == ARG
    assert lib.mt_exclusive_scan(A, B, S, N, I32, -1, None) == ARG
    assert lib.mt_exclusive_scan(None, B, S, N, I32, 0, None) == ARG
    assert lib.mt_exclusive_scan(A, B, None, N, I32, 0, None) == ARG
    assert lib.mt_exclusive_scan(A, B, S, None, I32, 0, None) == ARG
    assert lib.mt_exclusive_scan(A, A, S, N, I32, 0, None) == ALIAS
    assert lib.mt_exclusive_scan(A + 4, B, S, N, I64, 0, None) == ALIGN
    assert lib.mt_exclusive_scan(A, B, S + 8, N, I32, 0, None) == ALIGN
    assert lib.mt_exclusive_scan(A, B, S, N + 2, I32, 0, None) == ALIGN


def test_inclusive_scan_and_reduce_host_checks(lib):
    for fn in (lib.mt_inclusive_scan, lib.mt_reduce):
        assert fn(A, B, S, N, BF16, 0, None) == DTYPE
        assert fn(A, B, S, N, I32, 3, None) == ARG
        assert fn(None, B, S, N, I32, 0, None) == ARG
        assert fn(A, B, None, N, I32, 0, None) == ARG
        assert fn(A, B, S, None, I32, 0, None) == ARG
        assert fn(A + 4, B, S, N, I64, 0, None) == ALIGN
        assert fn(A, B, S, N + 2, I32, 0, None) == ALIGN


def test_select_host_checks(lib):
    assert lib.mt_select(None, A, B, N, S, N, None) == ARG
    assert lib.mt_select(A, B, A, N, S, N, None) == ALIAS
    assert lib.mt_select(A + 2, B, S, N, S, N, None) == ALIGN
    assert lib.mt_select(A, B, S, N + 1, S, N, None) == ALIGN


def test_select_wide_host_checks(lib):
    f = lib.mt_select_wide
    assert f(A, B, S, N, S, N, 3, None) == ARG
    assert f(A, B, S, N, S, N, 0, None) == ARG
    assert f(A, B, S, N, S, N, 6, None) == ARG    # structs are whole 32-bit words
    assert f(A, B, S, N, S, N, 260, None) == ARG  # at most 64 words
    assert f(A + 2, B, S, N, S, N, 12, None) == ALIGN  # structs: 4-byte aligned arr
    assert f(A, B, A, N, S, N, 8, None) == ALIAS
    assert f(A + 4, B, S, N, S, N, 8, None) == ALIGN  # 8-byte elements: arr 8-byte aligned
    assert f(A, B, S + 4, N, S, N, 8, None) == ALIGN  # ... and out
    # (any 8-byte-aligned arr and any flags offset pass these checks: the GPU tests cover them)


def test_reduce_by_key_host_checks(lib):
    f = lib.mt_reduce_by_key_add
    C, D = 0x50000, 0x60000
    assert f(A, B, C, D, N, S, N, I64, I32, None) == DTYPE
    assert f(A, B, C, D, N, S, N, I32, BF16, None) == DTYPE
    assert f(None, B, C, D, N, S, N, I32, I32, None) == ARG
    assert f(A, B, A, D, N, S, N, I32, I32, None) == ALIAS
    assert f(A, B, C, B, N, S, N, I32, I32, None) == ALIAS
    assert f(A + 4, B, C, D, N, S, N, I32, I32, None) == ALIGN  # keys and values out of phase
    assert f(A + 2, B + 2, C, D, N, S, N, I32, I32, None) == ALIGN


def test_scratch_slots(lib):
    f = lib.mt_scan_scratch_slots
    assert f(0, I32, 1) == 4
    assert f(-1, I32, 1) == -1
    assert f(10, BF16, 1) == -1
    assert f(10, I32, 7) == -1
    # 12288 elements per super-tile for 4-byte types; every record is sixteen
    # 8-byte slots (one 128-byte line); up to three elements of head misalignment
    assert f(12288, I32, 1) == 4 + 16 * 2
    assert f(12285, F32, 1) == 4 + 16 * 1
    assert f(1 << 28, I32, 1) == 4 + 16 * 21846
    # 6144 elements per super-tile for i64
    assert f(6144, I64, 1) == 4 + 16 * 2
    assert f(6143, I64, 1) == 4 + 16 * 1
    # u32 as i32; u64 as i64
    assert f(12288, 5, 1) == 4 + 16 * 2 and f(6144, 6, 1) == 4 + 16 * 2
    # f64: runs of 13 chunks per thread, 256 x 13 x 2 = 6656 elements per tile
    assert f(6655, 7, 1) == 4 + 16 and f(6656, 7, 1) == 4 + 16 * 2
    # select: 8192 flags per tile
    assert f(1 << 28, I32, 2) == 4 + 16 * (1 << 15)
    assert f(1, I32, 2) == 4 + 16 * 1
    # reduce: a header and one partial slot per CTA, whatever the capacity
    assert f(1 << 28, I32, 3) == f(0, F32, 3) == f(5, I64, 3) == f(7, 7, 3) == 4 + 2 * 4096
    assert f(10, BF16, 3) == -1
    # reduce by key: 6144 elements per super-tile (plus up to 3 of head phase)
    assert f(6141, 0, 4) == 4 + 16 and f(6142, 0, 4) == 4 + 32 and f(0, 0, 4) == 4


def test_rows_scratch_slots(lib):
    """Workspace of the row scans: header + rows x tiles per row x one
    128-byte record, for the worse of the two row-start alignments."""
    lib.mt_scan_rows_scratch_slots.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    lib.mt_scan_rows_scratch_slots.restype = ctypes.c_int64
    f = lib.mt_scan_rows_scratch_slots
    assert f(0, 5, F32) == 0 and f(5, 0, BF16) == 0
    assert f(-1, 5, F32) == -1 and f(1, -5, F32) == -1 and f(1, 5, I32) == -1
    # rows that fit one CTA take none
    assert f(1024, 4096, F32) == 0 and f(8192, 8192, BF16) == 0 and f(4096, 4099, F16) == 0
    # 16384 f32 fit one CTA from a 16-byte boundary, but not from off it: then
    # two tiles of 12288 (virtual) elements
    assert f(1, 16384, F32) == 4 + 16 * 2
    # long rows: 12288 f32 / 16384 bf16 elements per tile, up to 3 / 7 of head
    assert f(4, 1 << 24, F32) == 4 + 4 * 1366 * 16
    assert f(1, 1 << 24, BF16) == 4 + 1025 * 16 and f(3, 1 << 24, F16) == 4 + 3 * 1025 * 16
    assert f(1 << 40, 1 << 40, F32) == -1  # overflow


def test_strerror_and_counter(lib):
    assert lib.mt_scan_strerror(0) == b"ok"
    assert b"look-back" in lib.mt_scan_strerror(TIMEOUT)
    assert lib.mt_scan_strerror(12345) == b"unknown status"
    assert lib.mt_scan_launches() == 0  # nothing was launched on the CPU


def test_package_fails_loudly_without_library():
    """With the shared library absent the package refuses to import (no fallback)."""
    with tempfile.TemporaryDirectory() as d:
        pkg = os.path.join(d, "prefix_scan_row_gb300")
        os.makedirs(pkg)
        shutil.copy(os.path.join(ROOT, "prefix_scan_row_gb300", "__init__.py"), pkg)
        r = subprocess.run([sys.executable, "-c", "import prefix_scan_row_gb300"], cwd=d,
                           capture_output=True, text=True)
        assert r.returncode != 0
        assert "no CPU fallback" in r.stderr


def test_product_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "prefix_scan_row_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read().lower()
                assert "oracle" not in text, f
