"""Benchmark of the scan library on one GB300 (or N, one process per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the row-wise scan over the bf16/f16 workload:
[8192, 8192] exclusive and [4096, 4099] inclusive, each in bf16 and f16
storage (N(0, 1) inputs, seed 1), f32 accumulation -- four mt_scan_rows calls.
The metric is algorithmic HBM bytes (one read and one write of every element
in its storage width) per second, in GB/s. Inputs are resident in HBM when
the timed region starts; one step moves 671 MB, more than the 129 MB L2, and
no buffer is touched twice within a step, so nothing is served from L2
across iterations.

Printed: one JSON line (rank 0). Besides the device-timed value it carries
`e2e` (the same metric through the C ABI with host buffers: pinned host ->
device copy, the four calls, device -> host copy, every step), `roofline` for
the dominant kernel (the [8192, 8192] bf16 launch), `cpu_baseline` (the CPU
oracle, single-threaded, on a bounded sample), `clocks` sampled during the
timed region and `gpu_launches` counted by the library.

`--impl reference` times the CPU oracle instead (the only reference this
library has), on the same workload, metric and unit.

With N > 1 (torchrun), every rank runs the same per-GPU workload (weak
scaling: rows are independent and shard with no exchange); the time is the
max over ranks and the value the bytes of all ranks over that time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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

# (name, rows, n, storage dtype, inclusive); the first is the dominant launch
CALLS = [
    ("bf16_8192x8192_excl", 8192, 8192, "bf16", False),
    ("f16_8192x8192_excl", 8192, 8192, "f16", False),
    ("bf16_4096x4099_incl", 4096, 4099, "bf16", True),
    ("f16_4096x4099_incl", 4096, 4099, "f16", True),
]
DOMINANT = CALLS[0][0]
WORKLOAD = ("row-wise sum scan, bf16 and f16 storage with f32 accumulation: "
            "[8192,8192] exclusive + [4096,4099] inclusive (ragged, misaligned rows), "
            "iid N(0,1) seed 1; one step = the 4 calls")


def call_bytes(rows, n, dtype):
    return 2 * rows * n * (4 if dtype == "f32" else 2)


STEP_BYTES = sum(call_bytes(r, n, d) for _, r, n, d, _ in CALLS)
STEP_ELEMS = sum(r * n for _, r, n, _, _ in CALLS)
DOM_BYTES = call_bytes(*CALLS[0][1:4])

KERNEL_SOURCES = ["prefix_scan_row_gb300/csrc/mt_tile.cuh", "prefix_scan_row_gb300/csrc/mt_lookback.cuh",
                  "prefix_scan_row_gb300/csrc/mt_tilescan.cuh", "prefix_scan_row_gb300/csrc/mt_rows.cu"]
PROFILE = "profiles/rows_bf16_8192x8192_excl.md"


def kernel_source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when that summary was taken on other kernel sources."""
    try:
        text = open(os.path.join(ROOT, PROFILE)).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return int(m.group(1))


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
