"""Benchmark of the scan library on one GB300 (or N, one process per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is the device-wide 1-D exclusive scan workload, the largest of the
library's configured workloads: capacity 2^28 with a live count
n = 2^28 - 12345 held in device memory, i32 values uniform in [0, 15], f32
uniform[-1, 1) and i64 uniform in [0, 2^20) (seed 3), and exclusive_scan
add, min and max of each -- nine mt_exclusive_scan calls (each a status reset
kernel and the single-pass scan kernel), 25.77 GB of algorithmic traffic.
The metric is algorithmic HBM bytes (one read and one write of every live
element in its storage width) per second, in GB/s. Inputs are resident in HBM
when the timed region starts; every call moves 2.1 or 4.3 GB, many times the
129 MB L2, so nothing is served from L2 across calls.

Printed: one JSON line (rank 0). Besides the device-timed value it carries
`e2e` (the same step through the C ABI from pinned host buffers: host ->
device copy of the inputs, the nine calls, device -> host copy of the nine
results, every step), `roofline` for the dominant kernel (the i64 add scan),
`kernels` (every scan kernel on its configured workload: rows, long rows, the
nine 1-D scans and select at both densities, each timed back to back over
buffer sets larger than twice the L2), `cpu_baseline` (the CPU oracle, one
thread), `cpu_all_cores` (an all-core C scan, a second baseline), `clocks`
sampled during the timed region and `gpu_launches` counted by the library.

`--impl reference` times the CPU oracle instead (the only reference this
library has), on the same workload, metric and unit.

With N > 1 (torchrun), every rank runs the same per-GPU workload (weak
scaling: the replicas are independent, no data crosses ranks); the time is
the max over ranks and the value the bytes of all ranks over that time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "scan GB/s (read+write) and fraction of GB300 HBM peak; elements/s"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1000 * 1000

N_LIVE = workloads.SCAN1D_LIVE
CAPACITY = workloads.SCAN1D_CAPACITY
DTYPES = ("i32", "f32", "i64")
OPS = ("add", "min", "max")
SIZE = {"i32": 4, "f32": 4, "i64": 8, "bf16": 2, "f16": 2}
TORCH_DT = {"i32": torch.int32, "f32": torch.float32, "i64": torch.int64}
# (dtype, op) of the step's calls, in launch order
CALLS = [(d, op) for d in DTYPES for op in OPS]
DOMINANT = ("i64", "add")
WORKLOAD = ("device-wide 1-D exclusive_scan add/min/max: capacity 2^28, live count n = 2^28-12345 in "
            "device memory; i32 uniform in [0,15], f32 uniform[-1,1), i64 uniform in [0,2^20), seed 3; "
            "one step = the 9 calls (3 dtypes x 3 ops)")


def scan_bytes(dtype, n=N_LIVE):
    return 2 * SIZE[dtype] * n


def call_bytes(rows, n, dtype):
    return 2 * rows * n * SIZE[dtype]


STEP_BYTES = sum(scan_bytes(d) for d, _ in CALLS)
STEP_ELEMS = N_LIVE * len(CALLS)
DOM_BYTES = scan_bytes(DOMINANT[0])
B2B_LAUNCHES = 20  # back-to-back calls per kernel entry

# Sources of each kernel family: a profile's counters hold while these are
# unchanged (each sidecar in profiles/ stores the hash it was captured on).
_CSRC = "prefix_scan_row_gb300/csrc/"
FAMILY_SOURCES = {
    "rows": ["mt_internal.h", "mt_tile.cuh", "mt_lookback.cuh", "mt_tilescan.cuh", "mt_rows.cuh", "mt_rows.cu",
             "mt_staged.cuh"],
    "scan1d": ["mt_internal.h", "mt_tile.cuh", "mt_lookback.cuh", "mt_staged.cuh", "mt_scan1d.cuh", "mt_scan1d.cu"],
    "select": ["mt_internal.h", "mt_tile.cuh", "mt_lookback.cuh", "mt_select.cu"],
    "reduce": ["mt_internal.h", "mt_tile.cuh", "mt_reduce.cu"],
    "rbk": ["mt_internal.h", "mt_tile.cuh", "mt_lookback.cuh", "mt_rbk.cu"],
}


def _code_only(text):
    """A source file without its comments and blank lines: an edit of a
    comment leaves the hash (and the counters it vouches for) unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(family):
    h = hashlib.sha256()
    for p in FAMILY_SOURCES[family]:
        with open(os.path.join(ROOT, _CSRC + p), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(profile, family):
    """Per-launch DRAM bytes (read + write) of a kernel from its ncu sidecar
    (profiles/<name>.json), or None when there is none or it was captured on
    other kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", profile + ".json")) as f:
            side = json.load(f)
    except (OSError, ValueError):
        return None
    if side.get("kernel_source_hash") != kernel_source_hash(family):
        return None
    t = side.get("traffic_bytes_per_launch")
    return int(t) if t is not None else None


# ---------------------------------------------------------------------------
# SM clocks and clock-event reasons, sampled during the timed region (NVML
# through ctypes). Read-only.
# ---------------------------------------------------------------------------
_REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
            0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []  # (t, sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + bus)
            self._ct, self._nvml, self._handle = ctypes, nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            self._nvml = None

    def _run(self):
        ct, nv, h = self._ct, self._nvml, self._handle
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            ok = nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0
            ok2 = self._reasons_fn(h, ct.byref(rs)) == 0
            if ok:
                self.samples.append((time.perf_counter(), int(mhz.value), int(rs.value) if ok2 else 0))
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "sampled inside the timed region"
        if len(inside) < 3:  # a very short timed region: widen to the nearest samples
            inside = [s for s in self.samples if t0 - 0.3 <= s[0] <= t1 + 0.3]
            note = "timed region shorter than 3 samples; samples within 0.3 s of it"
        reasons = set()
        for _, _, m in inside:
            for bit, name in _REASONS.items():
                if m & bit:
                    reasons.add(name)
        reasons.discard("gpu_idle")
        return {"sm_mhz": statistics.median([s[1] for s in inside]) if inside else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons), "samples": len(inside),
                "source": "nvml" if self._nvml is not None else "unavailable", "note": note}


# ---------------------------------------------------------------------------
# Ranks (torchrun) -- one process per GPU, no data-path collective.
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(ms_local: float, bytes_local: float, device=None):
    """(max over ranks of the time, sum over ranks of the bytes). Works with
    any initialised process group (nccl on GPUs, gloo on CPU)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return ms_local, bytes_local
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    b = torch.tensor([bytes_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the --impl reference arm)
# ---------------------------------------------------------------------------
def make_host_inputs():
    """The step's three input arrays (the whole capacity), on the host."""
    return {d: workloads.scan1d(d) for d in DTYPES}


def oracle_sample(host, m):
    """The oracle's exclusive scan of the first m live elements of each of the
    step's nine calls. Returns (seconds, algorithmic bytes, elements)."""
    import oracle
    secs = nbytes = 0
    for d, op in CALLS:
        t = time.perf_counter()
        oracle.exclusive_scan(host[d], m, d, op)
        secs += time.perf_counter() - t
        nbytes += scan_bytes(d, m)
    return secs, nbytes, m * len(CALLS)


def calibrate_oracle(host):
    """Seconds one full step takes on the oracle, from a small sample."""
    m = 1 << 21
    secs, nbytes, _ = oracle_sample(host, m)
    return secs * STEP_BYTES / nbytes


def cpu_baseline(host, target_s=12.0):
    per_step = calibrate_oracle(host)
    m = min(N_LIVE, max(1 << 20, int(N_LIVE * target_s / per_step)))
    secs, nbytes, elems = oracle_sample(host, m)
    return {"value": nbytes / secs / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "elements_per_s": elems / secs, "seconds": round(secs, 3),
            "sample": f"the first {m} live elements of each of the step's 9 calls ({elems} elements, "
                      f"{nbytes} algorithmic bytes), plain C oracle, 1 thread"}


def cpu_all_cores(host, reps=3):
    """A second CPU baseline: the step's nine exclusive scans by an all-core C
    scan (pthreads, two-pass blocked; baselines/cpu_allcore.c), median of
    `reps` whole steps. Not the oracle, and not a target."""
    import numpy as np

    from baselines import allcore
    cores = allcore.cores()
    outs = {d: np.empty(host[d].shape, dtype=host[d].numpy().dtype) for d in DTYPES}
    times = []
    for _ in range(reps + 1):
        t0 = time.perf_counter()
        for d, op in CALLS:
            allcore.exclusive_scan(host[d], N_LIVE, d, op, cores, out=outs[d])
        times.append(time.perf_counter() - t0)
    secs = statistics.median(times[1:])  # the first pass pages the buffers in
    return {"value": STEP_BYTES / secs / 1e9, "unit": UNIT, "cores": cores,
            "kind": "all-core C exclusive scan (pthreads, two-pass blocked); a baseline, not the oracle",
            "elements_per_s": STEP_ELEMS / secs, "seconds_per_step": round(secs, 4),
            "sample": f"the whole step (9 calls, {STEP_ELEMS} elements), median of {reps}"}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
class Scan1D:
    """Device buffers of the step: one input, one output and one scratch per
    dtype, and the live count in device memory."""

    def __init__(self, mt, host, dev):
        self.mt = mt
        self.arr = {d: host[d].to(dev) for d in DTYPES}
        self.out = {d: torch.empty_like(self.arr[d]) for d in DTYPES}
        self.scratch = {d: mt.alloc_scratch(CAPACITY, TORCH_DT[d], mt.MT_SCRATCH_SCAN, device=dev) for d in DTYPES}
        self.n_dev = torch.tensor([N_LIVE], dtype=torch.int32, device=dev)

    def call(self, d, op, stream, out=None):
        self.mt.mt_exclusive_scan(self.arr[d], self.out[d] if out is None else out, self.scratch[d], self.n_dev,
                                  op, stream)

    def step(self, stream):
        for d, op in CALLS:
            self.call(d, op, stream)


def back_to_back(fns, stream, launches=B2B_LAUNCHES):
    """Average milliseconds per call of `fns` (closures over distinct buffer
    sets, together larger than twice the L2) called round-robin back to back
    between one event pair, after one warm-up round."""
    for f in fns:
        f()
    rounds = max(1, math.ceil(launches / len(fns)))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(rounds):
        for f in fns:
            f()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / (rounds * len(fns)), rounds * len(fns)


def graph_back_to_back(fns, launches):
    """The same as back_to_back for calls of a few microseconds: the calls
    (each takes the stream to enqueue on) are captured once, round-robin, in
    one CUDA graph on a side stream, and the graph is replayed between one
    event pair after one warm-up replay, so each launch costs the GPU's own
    scheduling and not a host submission."""
    side = torch.cuda.Stream()
    rounds = max(1, math.ceil(launches / len(fns)))
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        for f in fns:  # warm-up outside the capture
            f(side)
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(rounds):
                for f in fns:
                    f(side)
        g.replay()
        side.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(side)
        g.replay()
        b.record(side)
        b.synchronize()
    del g
    return a.elapsed_time(b) / (rounds * len(fns)), rounds * len(fns)


GRAPH_TIMING = ("calls captured round-robin in one CUDA graph and replayed between one event pair after a "
                "warm-up replay (calls under 256 MB, a few microseconds each)")


def kernel_entry(kernel, workload, nbytes, ms, launches, sets, peak, profile, family, **extra):
    achieved = nbytes / (ms / 1e3) / 1e9
    e = {"kernel": kernel, "workload": workload, "bound": "hbm", "bytes_per_launch": int(nbytes),
         "avg_launch_ms": round(ms, 5), "achieved": round(achieved, 1), "peak": peak, "unit": UNIT,
         "frac": round(achieved / peak, 4),
         "traffic": profile_traffic(profile, family) if profile else None,
         "profile": f"profiles/{profile}.json" if profile else None, "launches_timed": launches, "buffer_sets": sets}
    e.update(extra)
    return e


def launches_for(nbytes):
    """Back-to-back launches of a kernel entry: calls under 256 MB (tens of
    microseconds each) take ten times as many, so each entry times a few
    milliseconds of work at least."""
    return B2B_LAUNCHES if nbytes >= (256 << 20) else 10 * B2B_LAUNCHES


def sets_for(nbytes):
    """Buffer sets whose bytes together exceed twice the L2."""
    return max(1, -(-2 * L2_BYTES // nbytes))


def measure_kernels(mt, s1d, stream, dev, peak):
    """Every kernel on its configured workload (the scans, long rows and
    select), and the struct select, the reduction and reduce-by-key on the
    suite's workloads, each timed back to back after the main timed region
    (see back_to_back)."""
    ks = {}
    for d, op in CALLS:
        ms, n = back_to_back([lambda d=d, op=op: s1d.call(d, op, stream)], stream)
        name = f"exclusive_scan_{d}_{op}"
        ks[name] = kernel_entry(
            f"k_scan_staged ({d}, {op})", f"1-D exclusive scan {d} {op}, n = 2^28-12345 (capacity 2^28)",
            scan_bytes(d), ms, n, 1, peak, f"scan1d_{d}_{op}", "scan1d",
            note="each call is a status-reset launch plus the scan launch; the time covers both")
    # row scans: f32 [1024, 4096] (seed 0), bf16/f16 [8192, 8192] exclusive and
    # [4096, 4099] inclusive (seed 1), long rows f32 [4, 2^24] (seed 2)
    rows_cases = [
        ("rows_f32_1024x4096_incl", "k_scan_rows (f32)", "row scan f32 [1024,4096] inclusive", 1024, 4096, "f32", True),
        ("rows_f32_1024x4096_excl", "k_scan_rows (f32)", "row scan f32 [1024,4096] exclusive", 1024, 4096, "f32", False),
        ("rows_bf16_8192x8192_excl", "k_scan_rows (bf16)", "row scan bf16 [8192,8192] exclusive", 8192, 8192, "bf16",
         False),
        ("rows_f16_8192x8192_excl", "k_scan_rows (f16)", "row scan f16 [8192,8192] exclusive", 8192, 8192, "f16", False),
        ("rows_bf16_4096x4099_incl", "k_scan_rows (bf16)", "row scan bf16 [4096,4099] inclusive (ragged rows)", 4096,
         4099, "bf16", True),
        ("rows_f16_4096x4099_incl", "k_scan_rows (f16)", "row scan f16 [4096,4099] inclusive (ragged rows)", 4096,
         4099, "f16", True),
        ("rows_f32_4x2p24_incl", "k_scan_staged (long rows, f32)", "long-row scan f32 [4,2^24] inclusive", 4, 1 << 24,
         "f32", True),
        ("rows_f32_4x2p24_excl", "k_scan_staged (long rows, f32)", "long-row scan f32 [4,2^24] exclusive", 4, 1 << 24,
         "f32", False),
    ]
    half = {}
    for name, kern, wl, r, n, d, inc in rows_cases:
        if d == "f32":
            x = (workloads.rows_f32(r, n) if r == 1024 else workloads.rows_long(r, n)).to(dev)
        else:
            x = half.get((r, n, d))
            if x is None:
                x = half[(r, n, d)] = workloads.rows_half(r, n, d).to(dev)
        nb = call_bytes(r, n, d)
        sets = sets_for(nb)
        xs = [x] + [x.clone() for _ in range(sets - 1)]
        os_ = [torch.empty_like(x) for _ in range(sets)]
        if nb < (256 << 20):  # single-tile rows: no allocation, capturable
            fns = [lambda st, xi=xi, oi=oi: mt.mt_scan_rows(xi, oi, inc, st) for xi, oi in zip(xs, os_)]
            ms, nl = graph_back_to_back(fns, launches_for(nb))
            ks[name] = kernel_entry(kern, wl, nb, ms, nl, sets, peak, name, "rows", timing=GRAPH_TIMING)
        else:
            fns = [lambda xi=xi, oi=oi: mt.mt_scan_rows(xi, oi, inc, stream) for xi, oi in zip(xs, os_)]
            ms, nl = back_to_back(fns, stream, launches_for(nb))
            ks[name] = kernel_entry(kern, wl, nb, ms, nl, sets, peak, name, "rows")
        del xs, os_, fns
    # the four row calls of the bf16/f16 workload as one sequence
    seq = [(8192, 8192, "bf16", False), (8192, 8192, "f16", False), (4096, 4099, "bf16", True),
           (4096, 4099, "f16", True)]
    outs = [torch.empty_like(half[(r, n, d)]) for r, n, d, _ in seq]
    fns = [lambda st, x=half[(r, n, d)], o=o, inc=inc: mt.mt_scan_rows(x, o, inc, st)
           for (r, n, d, inc), o in zip(seq, outs)]
    nb = sum(call_bytes(r, n, d) for r, n, d, _ in seq) / len(seq)
    ms, nl = graph_back_to_back(fns, launches_for(nb))
    ks["rows_half_4_calls"] = kernel_entry(
        "k_scan_rows (bf16, f16)", "bf16 and f16 [8192,8192] exclusive then [4096,4099] inclusive, in turn", nb, ms,
        nl, 1, peak, None, "rows", timing=GRAPH_TIMING,
        note="bytes_per_launch and avg_launch_ms are the means over the four calls")
    del half, outs, fns
    # select: f32 values n = 2^28 uniform[-1,1) (seed 4), u8 flags Bernoulli(p) (seed 5)
    ns = workloads.SELECT_N
    vals = workloads.uniform((ns,), workloads.SEED_SELECT, -1.0, 1.0, "f32").to(dev)
    out = torch.empty_like(vals)
    num = torch.zeros(1, dtype=torch.int32, device=dev)
    scr = mt.alloc_scratch(ns, torch.int32, mt.MT_SCRATCH_SELECT, device=dev)
    nd = torch.tensor([ns], dtype=torch.int32, device=dev)
    for p, tag in ((0.5, "p05"), (0.01, "p001")):
        flags = workloads.bernoulli_u8(ns, p, workloads.SEED_SELECT + 1).to(dev)
        k = int(flags.sum().item())
        ms, nl = back_to_back([lambda f=flags: mt.mt_select(vals, f, out, num, scr, nd, stream)], stream)
        ks[f"select_f32_{tag}"] = kernel_entry(
            "k_select_staged (4-byte values)", f"select f32, n = 2^28, flags Bernoulli(p = {p})", 5 * ns + 4 * k, ms,
            nl, 1, peak, f"select_f32_{tag}", "select", selected=k,
            note="bytes_per_launch = 5 n + 4 num_out (flags and values read, selected values written); each call "
                 "is a status-reset launch plus the select launch")
        del flags
    # select of 12-byte structs (k_select_words<3>): the f32 values above as
    # the first word of each struct, p = 0.5
    flags = workloads.bernoulli_u8(ns, 0.5, workloads.SEED_SELECT + 1).to(dev)
    k = int(flags.sum().item())
    v3 = vals.view(torch.int32).unsqueeze(1).expand(ns, 3).contiguous()
    del out
    o3 = torch.empty_like(v3)
    ms, nl = back_to_back([lambda: mt.mt_select_wide(v3, flags, o3, num, scr, nd, stream)], stream)
    ks["select_struct12_p05"] = kernel_entry(
        "k_select_words<3> (12-byte structs)", "select of 12-byte structs, n = 2^28, flags Bernoulli(p = 0.5)",
        13 * ns + 12 * k, ms, nl, 1, peak, "select_struct12_p05", "select", selected=k,
        note="bytes_per_launch = 13 n + 12 num_out by the select formula (flags and structs read, selected "
             "structs written); each call is a status-reset launch plus the select launch")
    del v3, o3, flags, vals, scr
    # reduce: i32 add over the step's i32 input (n = 2^28 - 12345), read only
    rscr = mt.alloc_scratch(CAPACITY, torch.int32, mt.MT_SCRATCH_REDUCE, device=dev)
    r1 = torch.empty(1, dtype=torch.int32, device=dev)
    ms, nl = back_to_back([lambda: mt.mt_reduce(s1d.arr["i32"], r1, rscr, s1d.n_dev, "add", stream)], stream)
    ks["reduce_i32_add"] = kernel_entry(
        "k_reduce (i32, add)", "reduce i32 add, n = 2^28-12345 (the step's i32 input)", 4 * N_LIVE, ms, nl, 1, peak,
        "reduce_i32_add", "reduce",
        note="bytes_per_launch = 4 n, read only, against the read+write copy peak; each call is a reset launch "
             "plus the reduce launch")
    del rscr, r1
    # reduce by key: n = 2^28 i32 keys in runs of geometric length (mean 8,
    # keys from an alphabet of 64), f32 values (seed 11)
    kk, vv = workloads.runs(ns, 8.0, workloads.SEED_SELECT + 7, "i32", "f32")
    kk, vv = kk.to(dev), vv.to(dev)
    ko, vo = torch.empty_like(kk), torch.empty_like(vv)
    bscr = mt.alloc_scratch(ns, torch.int32, mt.MT_SCRATCH_REDUCE_BY_KEY, device=dev)
    mt.mt_reduce_by_key_add(kk, vv, ko, vo, num, bscr, nd, stream)
    torch.cuda.synchronize()
    runs_n = int(num.item())
    ms, nl = back_to_back([lambda: mt.mt_reduce_by_key_add(kk, vv, ko, vo, num, bscr, nd, stream)], stream)
    ks["reduce_by_key_i32_f32"] = kernel_entry(
        "k_reduce_by_key (i32 keys, f32 values)",
        "reduce_by_key_add, n = 2^28, i32 keys in runs of geometric length (mean 8), f32 values",
        8 * ns + 8 * runs_n, ms, nl, 1, peak, "reduce_by_key_i32_f32", "rbk", runs=runs_n,
        note="bytes_per_launch = 8 n + 8 runs (keys and values read, one key and one sum written per run); each "
             "call is a reset launch plus the reduce-by-key launch")
    del kk, vv, ko, vo, bscr
    torch.cuda.synchronize()
    assert mt.mt_scan_status(stream) == 0, "device error word set while timing the kernels"
    return ks


def run_ours(args, world, rank, local):
    import prefix_scan_row_gb300 as mt
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    host = make_host_inputs()
    s1d = Scan1D(mt, host, dev)

    for _ in range(args.warmup):
        s1d.step(stream)
    torch.cuda.synchronize()
    assert mt.mt_scan_status(stream) == 0
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local).start()
    time.sleep(0.05)
    barrier()
    torch.cuda.synchronize()
    l0 = mt.mt_scan_launches()
    th0 = time.perf_counter()
    start.record(stream)
    for _ in range(args.steps):
        s1d.step(stream)
    end.record(stream)
    torch.cuda.synchronize()
    th1 = time.perf_counter()
    barrier()
    launches = mt.mt_scan_launches() - l0
    assert mt.mt_scan_status(stream) == 0, "device error word set during the timed region"
    ms_local = start.elapsed_time(end)
    ms, nbytes = aggregate(ms_local, STEP_BYTES * args.steps, dev if world > 1 else None)
    peak, peak_src = measured_peak()

    # The dominant kernel (the i64 add scan, the largest call of the step),
    # timed back to back after the timed region, then every other kernel on
    # its own workload.
    tk0 = time.perf_counter()
    dom_ms, dom_n = back_to_back([lambda: s1d.call(*DOMINANT, stream)], stream)
    kernels = measure_kernels(mt, s1d, stream, dev, peak) if not args.no_kernels else {}
    tk1 = time.perf_counter()
    time.sleep(0.05)
    sampler.stop()

    # End to end through the C ABI from host buffers (run_e2e).
    if args.no_e2e:
        e2e_line = None
    else:
        e2e_line = run_e2e(args, s1d, host, stream, dev, world)
    value = nbytes / (ms / 1e3) / 1e9
    achieved = DOM_BYTES / (dom_ms / 1e3) / 1e9
    line = make_line(args, world, value, ms, peak, peak_src, achieved, dom_ms, dom_n, kernels, sampler, th0, th1,
                     tk0, tk1, launches, e2e_line)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(host)
        line["cpu_all_cores"] = cpu_all_cores(host)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, s1d, host, stream, dev, world):
    """The e2e entry: the step through the C ABI from pinned host buffers.

    Every step copies the three inputs' live elements from pinned host memory
    to the device, makes the nine calls, and copies each call's result to its
    own pinned host buffer. Uploads run on one copy stream into two device
    input sets in turn and downloads on another, so a step's upload overlaps
    the previous step's downloads (the host link carries both directions at
    once) and each result's download overlaps the next call."""
    mt = s1d.mt
    pin_in = {d: host[d][:N_LIVE].pin_memory() for d in DTYPES}
    pin_out = [torch.empty(N_LIVE, dtype=TORCH_DT[d]).pin_memory() for d, _ in CALLS]
    dev_out = [torch.empty(N_LIVE, dtype=TORCH_DT[d], device=dev) for d, _ in CALLS]
    # two device input sets: the step's own buffers (rewritten with the same
    # values) and a second one of the same shape
    sets = [s1d.arr, {d: torch.empty_like(s1d.arr[d]) for d in DTYPES}]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = torch.cuda.Event
    loaded = [ev(), ev()]          # a set's inputs are on the device
    consumed = [ev(), ev()]        # a set's last call has read its inputs
    computed = [ev() for _ in CALLS]   # call i's result is written
    fetched = [ev() for _ in CALLS]    # call i's result has reached the host
    step_no = [0]

    def e2e_step():
        k = step_no[0]
        b = k % 2
        arr = sets[b]
        up.wait_event(consumed[b])  # the calls of step k - 2 are done with this set
        with torch.cuda.stream(up):
            for d in DTYPES:
                arr[d][:N_LIVE].copy_(pin_in[d], non_blocking=True)
        loaded[b].record(up)
        stream.wait_event(loaded[b])
        for i, (d, op) in enumerate(CALLS):
            stream.wait_event(fetched[i])  # the previous step's copy of this result is out
            mt.mt_exclusive_scan(arr[d], dev_out[i], s1d.scratch[d], s1d.n_dev, op, stream)
            computed[i].record(stream)
            down.wait_event(computed[i])
            with torch.cuda.stream(down):
                pin_out[i].copy_(dev_out[i], non_blocking=True)
            fetched[i].record(down)
        consumed[b].record(stream)
        step_no[0] += 1

    for e in consumed + fetched:
        e.record(stream)
    e2e_steps = max(1, min(args.steps, 5))
    e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_stream(down)
    stream.wait_stream(up)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    assert mt.mt_scan_status(stream) == 0
    e2e_ms, e2e_bytes = aggregate(e0.elapsed_time(e1), STEP_BYTES * e2e_steps, dev if world > 1 else None)
    h2d = sum(pin_in[d].numel() * pin_in[d].element_size() for d in DTYPES)
    d2h = sum(t.numel() * t.element_size() for t in pin_out)
    return {"value": round(e2e_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
            "how": "pinned host -> device copy of the 3 inputs' live elements (one copy stream, two device input "
                   "sets in turn), the 9 mt_exclusive_scan calls, device -> pinned host copy of each call's result "
                   "(a second copy stream); a step's upload overlaps the previous step's downloads; CUDA events "
                   "around the steps"}


def make_line(args, world, value, ms, peak, peak_src, achieved, dom_ms, dom_n, kernels, sampler, th0, th1, tk0,
              tk1, launches, e2e_line):
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i32+f32+i64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "calls_per_step": [f"exclusive_scan {d} {op}" for d, op in CALLS],
                   "live_n": N_LIVE, "capacity": CAPACITY, "bytes_per_step": STEP_BYTES,
                   "elements_per_step": STEP_ELEMS,
                   "l2": f"inputs larger than L2: each call moves {scan_bytes('i32') / 1e9:.2f} or "
                         f"{scan_bytes('i64') / 1e9:.2f} GB vs a {L2_BYTES / 1e6:.0f} MB L2",
                   "parallelism": f"replicas x{world} (independent problems, no exchange)"},
        "elements_per_s": round(STEP_ELEMS * world * args.steps / (ms / 1e3), 1),
        "frac_of_peak": {"measured": round(value / world / peak, 4), "peak_gbs": peak,
                         "peak_source": peak_src, "datasheet_8000_gbs": round(value / world / 8000.0, 4)},
        "e2e": e2e_line,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profile_traffic("scan1d_i64_add", "scan1d"),
                     "kernel": "k_scan_staged<long, OpAdd, 4, 3, 256> (1-D exclusive scan, i64 add)",
                     "bytes_per_launch": DOM_BYTES, "avg_launch_ms": round(dom_ms, 5), "timed_launches": dom_n,
                     "timing": f"{dom_n} calls back to back between one event pair after the timed region (each "
                               "call is a status-reset launch plus the scan launch; the time covers both)",
                     "peak_of": peak_src},
        "kernels": kernels,
        "clocks": sampler.summary(th0, th1),
        "clocks_kernels": sampler.summary(tk0, tk1),
        "gpu_launches": int(launches),
    }
    if e2e_line is None:
        del line["e2e"]
    return line


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle, as it stands, on the same workload.
# ---------------------------------------------------------------------------
def run_reference(args, world, rank):
    if rank != 0:
        return  # rank 0 alone runs the CPU reference
    host = make_host_inputs()
    per_step = calibrate_oracle(host)
    budget = 150.0  # seconds for the whole --warmup W --steps K run
    m = min(N_LIVE, max(1 << 16, int(N_LIVE * budget / max(1, args.steps + args.warmup) / per_step)))
    for _ in range(args.warmup):
        oracle_sample(host, m)
    secs = nbytes = elems = 0
    for _ in range(args.steps):
        s, b, e = oracle_sample(host, m)
        secs, nbytes, elems = secs + s, nbytes + b, elems + e
    value = nbytes / secs / 1e9
    sample = (f"each step: the first {m} live elements of each of the 9 calls ({m * len(CALLS)} elements), "
              f"plain C oracle, 1 thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs * 1e3 / max(1, args.steps), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "i32+f32+i64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "accumulate": "exact integers; f32 add in f64 (oracle)"},
        "elements_per_s": round(elems / secs, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# --suite: each kernel on each configured shape, one JSON line per call (not
# the bench line). Calls are timed one by one with CUDA events; L2 is flushed
# before every timed call whose buffers would fit in it.
# ---------------------------------------------------------------------------
def run_suite(args):
    import prefix_scan_row_gb300 as mt
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, src = measured_peak()
    # L2 flush by a read of twice its size: the lines left behind are clean,
    # so the timed call does not pay for writing back the flush's own data.
    flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    rows_out = []

    def wanted(name):
        return args.only is None or any(o in name for o in args.only.split("|"))

    def sustained(fns, nbytes, rounds=20):
        """Back-to-back calls rotating over buffer sets that together exceed
        twice the L2, between one event pair: the throughput of a stream of
        calls, each launch overlapping its neighbours' ramp and drain."""
        for f in fns:
            f()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(rounds):
            for f in fns:
                f()
        b.record()
        b.synchronize()
        ms = a.elapsed_time(b) / (rounds * len(fns))
        return nbytes / (ms / 1e3) / 1e9

    def timeit(name, fn, nbytes, elems, reps=20, rotate=None, touched=None):
        if not wanted(name):
            return
        small = nbytes < 2 * L2_BYTES
        for _ in range(3):
            fn()
        times = []
        for _ in range(reps):
            # The GPU is kept busy (an L2 flush, or a short sleep for inputs
            # larger than L2) while the host enqueues the call, so the events
            # time the call's kernels and not the host's launch latency.
            if small:
                flush.sum()
            else:
                torch.cuda._sleep(100_000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        assert mt.mt_scan_status() == 0
        med = statistics.median(times)
        gbs = nbytes / (med / 1e3) / 1e9
        r = {"config": name, "ms": round(med, 4), "GB/s": round(gbs, 1),
             "frac_measured": round(gbs / peak, 3), "frac_datasheet_8000_gbs": round(gbs / 8000.0, 3),
             "Gelem/s": round(elems / (med / 1e3) / 1e9, 2),
             "l2_flushed": small, "host_enqueue_hidden": True}
        if touched is not None:  # the bytes the launch actually moves (values read only when selected)
            tg = touched / (med / 1e3) / 1e9
            r.update({"touched_bytes": int(touched), "touched_GB/s": round(tg, 1),
                      "touched_frac_measured": round(tg / peak, 3)})
        if rotate is not None:
            sg = sustained(rotate, nbytes)
            r.update({"back_to_back_GB/s": round(sg, 1), "back_to_back_frac_measured": round(sg / peak, 3),
                      "back_to_back_buffer_sets": len(rotate)})
        rows_out.append(r)
        print(json.dumps(r), flush=True)

    for name, (r, n, d), incs in [
            ("rows f32 [1024,4096]", (1024, 4096, "f32"), (True, False)),
            ("rows bf16 [8192,8192]", (8192, 8192, "bf16"), (False,)),
            ("rows f16 [8192,8192]", (8192, 8192, "f16"), (False,)),
            ("rows bf16 [4096,4099]", (4096, 4099, "bf16"), (True,)),
            ("rows f16 [4096,4099]", (4096, 4099, "f16"), (True,)),
            ("rows f32 [4,2^24]", (4, 1 << 24, "f32"), (True, False))]:
        if not any(wanted(f"{name} {'incl' if i else 'excl'}") for i in incs):
            continue
        x = (workloads.rows_f32(r, n) if d == "f32" else workloads.rows_half(r, n, d)).to(dev)
        o = torch.empty_like(x)
        sets = -(-2 * L2_BYTES // call_bytes(r, n, d))  # buffer sets for the back-to-back figure
        xs = [x] + [x.clone() for _ in range(sets - 1)]
        os_ = [o] + [torch.empty_like(x) for _ in range(sets - 1)]
        for inc in incs:
            timeit(f"{name} {'incl' if inc else 'excl'}", lambda: mt.mt_scan_rows(x, o, inc),
                   call_bytes(r, n, d), r * n,
                   rotate=[lambda xi=xi, oi=oi: mt.mt_scan_rows(xi, oi, inc) for xi, oi in zip(xs, os_)])
        del x, o, xs, os_
    # the product / max / min row scans on the same shapes
    for name, (r, n, d), inc in [
            ("rows_op {} f32 [1024,4096] incl", (1024, 4096, "f32"), True),
            ("rows_op {} bf16 [8192,8192] excl", (8192, 8192, "bf16"), False),
            ("rows_op {} bf16 [4096,4099] incl", (4096, 4099, "bf16"), True),
            ("rows_op {} f32 [4,2^24] incl", (4, 1 << 24, "f32"), True)]:
        if not any(wanted(name.format(op)) for op in ("mul", "max", "min")):
            continue
        x = (workloads.rows_f32(r, n) if d == "f32" else workloads.rows_half(r, n, d)).to(dev)
        o = torch.empty_like(x)
        for op in ("mul", "max", "min"):
            timeit(name.format(op), lambda: mt.mt_scan_rows_op(x, o, op, inc), call_bytes(r, n, d), r * n)
        del x, o
    cap, n = workloads.SCAN1D_CAPACITY // args.scale, workloads.SCAN1D_LIVE // args.scale
    tag = "n=2^28-12345" if args.scale == 1 else f"n=(2^28-12345)/{args.scale}"
    n_dev = torch.tensor([n], dtype=torch.int32, device=dev)
    for d, tdt, s in (("i32", torch.int32, 4), ("f32", torch.float32, 4), ("i64", torch.int64, 8),
                      ("u32", torch.uint32, 4), ("u64", torch.uint64, 8), ("f64", torch.float64, 8)):
        if not any(wanted(f"{k} {d} {op} {tag}") for op in ("add", "min", "max")
                   for k in ("exclusive_scan", "inclusive_scan", "reduce")):
            continue
        a = workloads.scan1d(d, capacity=cap).to(dev).view(tdt)  # unsigned: a view of the signed twin
        o = torch.empty(a.shape, dtype=torch.int64 if s == 8 else torch.int32, device=dev).view(tdt)
        scr = mt.alloc_scratch(cap, tdt, mt.MT_SCRATCH_SCAN, device=dev)
        for op in ("add", "min", "max"):
            timeit(f"exclusive_scan {d} {op} {tag}",
                   lambda: mt.mt_exclusive_scan(a, o, scr, n_dev, op), 2 * s * n, n)
        for op in ("add", "min", "max"):
            timeit(f"inclusive_scan {d} {op} {tag}",
                   lambda: mt.mt_inclusive_scan(a, o, scr, n_dev, op), 2 * s * n, n)
        rscr = mt.alloc_scratch(cap, tdt, mt.MT_SCRATCH_REDUCE, device=dev)
        r1 = torch.empty(1, dtype=torch.int64 if s == 8 else torch.int32, device=dev).view(tdt)
        for op in ("add", "min", "max"):
            timeit(f"reduce {d} {op} {tag}",
                   lambda: mt.mt_reduce(a, r1, rscr, n_dev, op), s * n, n)
        del a, o, scr, rscr, r1
    ns = workloads.SELECT_N // args.scale
    nd = torch.tensor([ns], dtype=torch.int32, device=dev)
    for p in (0.5, 0.01):
        if not wanted(f"select f32 n={ns} p={p}"):
            continue
        v, f = workloads.select_inputs(ns, p)
        k = int(f.sum())
        v, f = v.to(dev), f.to(dev)
        o = torch.empty_like(v)
        num = torch.zeros(1, dtype=torch.int32, device=dev)
        scr = mt.alloc_scratch(ns, torch.int32, mt.MT_SCRATCH_SELECT, device=dev)
        timeit(f"select f32 n={ns} p={p}", lambda: mt.mt_select(v, f, o, num, scr, nd),
               5 * ns + 4 * k, ns)
        del v, f, o, scr
    for p in (0.5, 0.01):  # values 4 bytes past a 16-byte boundary, flags at the boundary
        if not wanted(f"select f32 misaligned n={ns} p={p}"):
            continue
        v, f = workloads.select_inputs(ns, p)
        k = int(f.sum())
        vb = torch.empty(ns + 4, dtype=torch.float32, device=dev)
        vm = vb[1:1 + ns]
        vm.copy_(v.to(dev))
        f = f.to(dev)
        o = torch.empty(ns, dtype=torch.float32, device=dev)
        num = torch.zeros(1, dtype=torch.int32, device=dev)
        scr = mt.alloc_scratch(ns, torch.int32, mt.MT_SCRATCH_SELECT, device=dev)
        timeit(f"select f32 misaligned n={ns} p={p}", lambda: mt.mt_select(vm, f, o, num, scr, nd),
               5 * ns + 4 * k, ns)
        del v, vb, vm, f, o, scr
    for p in (0.5, 0.01):  # 8-byte elements: the same flags, f64 values
        if not wanted(f"select_wide f64 n={ns} p={p}"):
            continue
        v, f = workloads.select_inputs(ns, p)
        k = int(f.sum())
        v, f = v.to(dev).to(torch.float64), f.to(dev)
        o = torch.empty_like(v)
        num = torch.zeros(1, dtype=torch.int32, device=dev)
        scr = mt.alloc_scratch(ns, torch.int32, mt.MT_SCRATCH_SELECT, device=dev)
        timeit(f"select_wide f64 n={ns} p={p}", lambda: mt.mt_select_wide(v, f, o, num, scr, nd),
               9 * ns + 8 * k, ns)
        del v, f, o, scr
    for words in (3, 4, 6, 8):  # struct elements (12- to 32-byte structs): flags staged, values read once selected
        for p in (0.5, 0.01):
            name = f"select_wide struct {4 * words}B n={ns} p={p}"
            if not wanted(name):
                continue
            v, f = workloads.select_inputs(ns, p)
            k = int(f.sum())
            v = v.to(dev).view(torch.int32).unsqueeze(1).expand(ns, words).contiguous()
            f = f.to(dev)
            o = torch.empty_like(v)
            num = torch.zeros(1, dtype=torch.int32, device=dev)
            scr = mt.alloc_scratch(ns, torch.int32, mt.MT_SCRATCH_SELECT, device=dev)
            # 32-byte sectors of arr holding part of a selected struct (the only value bytes read)
            sel = torch.nonzero(f).flatten().to(torch.int64)
            sec = torch.zeros((4 * words * ns + 31) // 32, dtype=torch.bool, device=dev)
            sec[(4 * words * sel) // 32] = True
            sec[(4 * words * sel + 4 * words - 1) // 32] = True
            touched = ns + 32 * int(sec.sum()) + 4 * words * k
            del sel, sec
            timeit(name, lambda: mt.mt_select_wide(v, f, o, num, scr, nd), (1 + 4 * words) * ns + 4 * words * k, ns,
                   touched=touched)
            del v, f, o, scr
    # reduce by key: i32 keys in runs of mean length 8, f32 values
    nr = workloads.SELECT_N // args.scale
    if wanted(f"reduce_by_key i32/f32 n={nr} mean_run=8"):
        kk, vv = workloads.runs(nr, 8.0, workloads.SEED_SELECT + 7, "i32", "f32")
        kk, vv = kk.to(dev), vv.to(dev)
        ko, vo = torch.empty_like(kk), torch.empty_like(vv)
        num = torch.zeros(1, dtype=torch.int32, device=dev)
        scr = mt.alloc_scratch(nr, torch.int32, mt.MT_SCRATCH_REDUCE_BY_KEY, device=dev)
        nrd = torch.tensor([nr], dtype=torch.int32, device=dev)
        mt.mt_reduce_by_key_add(kk, vv, ko, vo, num, scr, nrd)
        torch.cuda.synchronize()
        runs_n = int(num.item())
        timeit(f"reduce_by_key i32/f32 n={nr} mean_run=8",
               lambda: mt.mt_reduce_by_key_add(kk, vv, ko, vo, num, scr, nrd), 8 * nr + 8 * runs_n, nr)
        del kk, vv, ko, vo, scr
    if args.suite_out:
        with open(args.suite_out, "w") as fh:
            json.dump({"peak_gbs": peak, "peak_source": src, "rows": rows_out}, fh, indent=1)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the CPU baselines (profiling runs)")
    ap.add_argument("--no-kernels", action="store_true",
                    help="skip the per-kernel back-to-back entries (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg through host buffers (profiling runs)")
    ap.add_argument("--suite", action="store_true", help="time every kernel on every configured shape")
    ap.add_argument("--suite-out", default=None)
    ap.add_argument("--only", default=None, help="suite: run only configs whose name contains this")
    ap.add_argument("--scale", type=int, default=1, help="suite: divide the 1-D sizes by this")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_env()
    if args.suite:
        run_suite(args)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
