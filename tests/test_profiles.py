"""The ncu sidecars under profiles/ that bench.py reads for each kernel
entry's `traffic`: every entry has one, each parses, names its kernel family,
was taken on the family's current sources (a kernel changed since its
counters were taken must be re-captured, else the bench reports no traffic
for it), and its DRAM traffic is close to the entry's algorithmic bytes (far
above them would mean re-reads; an output still in L2 when the launch ends
only lowers the write count)."""
import json
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# every kernel entry of the bench line that names a sidecar
ENTRIES = ([f"scan1d_{d}_{op}" for d in ("i32", "f32", "i64") for op in ("add", "min", "max")]
           + ["rows_f32_1024x4096_incl", "rows_f32_1024x4096_excl", "rows_bf16_8192x8192_excl",
              "rows_f16_8192x8192_excl", "rows_bf16_4096x4099_incl", "rows_f16_4096x4099_incl",
              "rows_f32_4x2p24_incl", "rows_f32_4x2p24_excl",
              "select_f32_p05", "select_f32_p001", "select_struct12_p05", "reduce_i32_add",
              "reduce_by_key_i32_f32"])


def load(tag):
    with open(os.path.join(ROOT, "profiles", f"{tag}.json")) as f:
        return json.load(f)


def test_every_family_source_exists():
    for fam, files in bench.FAMILY_SOURCES.items():
        for p in files:
            assert os.path.isfile(os.path.join(ROOT, "prefix_scan_row_gb300", "csrc", p)), (fam, p)


@pytest.mark.parametrize("tag", ENTRIES)
def test_sidecar_is_current(tag):
    d = load(tag)
    fam = d["kernel_family"]
    assert fam in bench.FAMILY_SOURCES
    assert d["kernel_source_hash"] == bench.kernel_source_hash(fam), (
        f"profiles/{tag}.json was captured on other sources of the '{fam}' kernels: re-capture it")
    assert bench.profile_traffic(tag, fam) == d["traffic_bytes_per_launch"]


@pytest.mark.parametrize("tag", ENTRIES)
def test_sidecar_traffic_near_algorithmic_bytes(tag):
    d = load(tag)
    assert d["traffic_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    ratio = d["traffic_bytes_per_launch"] / d["algorithmic_bytes_per_launch"]
    # low: outputs that fit in L2 are mostly still there when the launch ends
    assert 0.4 < ratio < 1.05, (tag, ratio)
    assert d["duration_us_cold_serialised"] > 0


def test_dominant_kernel_sidecar_is_the_roofline_one():
    d = load("scan1d_i64_add")
    assert d["algorithmic_bytes_per_launch"] == bench.DOM_BYTES


def test_source_hash_ignores_comments_but_not_code():
    src = "int a = 1;  // one\n/* block\n   comment */\nint b = a + 2;\n"
    same = "int a = 1;  // another note\n\nint b = a + 2;   \n"
    changed = "int a = 1;\nint b = a + 3;\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(changed)
