"""Builds libmtscan.so in-tree for sm_103a (GB300), and its bounds-checked
twin libmtscan_checked.so.

Each .cu file is compiled by nvcc in parallel, then linked into one shared
library next to this file. The CUDA runtime is linked statically, so the
library loads without any library path set up. The checked library is the
same sources compiled with MT_CHECKED=1: every global store and shared-memory
access of its kernels is checked against its buffer first, and a bad one is
skipped and reported as MT_ERR_BOUNDS by mt_scan_status() (a debugging and
test build; the ordinary library is the product).
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmtscan.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmtscan_checked.so")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "mt_scan.h"))
    return max(os.path.getmtime(h) for h in hs)


def _variant(checked):
    return (BUILD_CHECKED, LIB_CHECKED, ["-DMT_CHECKED=1"]) if checked else (BUILD, LIB, [])


def _compile(src, extra, checked):
    bdir, _, defs = _variant(checked)
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    if (not extra and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime())):
        return obj
    cmd = [NVCC, *ARCH, *FLAGS, *defs, *extra, "-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def _link(objs, checked, force):
    _, lib, _ = _variant(checked)
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Builds one library (the checked twin with `checked`); returns its path."""
    return build_all(force, verbose_ptxas, variants=(checked,))[0]


def build_all(force: bool = False, verbose_ptxas: bool = False, variants=(False, True)):
    """Builds the ordinary and the checked library, every translation unit of
    both in one pool of compiler processes; returns their paths."""
    for checked in variants:
        bdir = _variant(checked)[0]
        os.makedirs(bdir, exist_ok=True)
        if force:
            for f in os.listdir(bdir):
                os.remove(os.path.join(bdir, f))
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    srcs = sources()
    jobs = [(src, checked) for checked in variants for src in srcs]
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], extra, j[1]), jobs))
    libs = []
    for i, checked in enumerate(variants):
        libs.append(_link(objs[i * len(srcs):(i + 1) * len(srcs)], checked, force))
    return libs


if __name__ == "__main__":
    print(*build_all(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv), sep="\n")
