"""The pins have teeth: each build of the oracle with one planted mistake (a
swapped boundary, a wrong sign, a dropped term, a wrong identity, a
transposed comparison or index, a wrong rounding rule) must fail at least one
pin. The mistakes are planted in a temporary copy of the oracle's C source on
the CPU; the real oracle is untouched."""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "mt_oracle.c")

MUTANTS = {
    "incl_excl_swapped": ("const double y = inclusive ? lp_next : lp;",
                          "const double y = inclusive ? lp : lp_next;"),
    "row_wrong_sign": ("const double lp_next = lp + x;", "const double lp_next = lp - x;"),
    "row_transposed_index": ("const int64_t k = r * n + i;", "const int64_t k = r + i * rows;"),
    "i32_dropped_first_term": ("lp += (uint32_t)x[i];", "if (i) lp += (uint32_t)x[i];"),
    "i32_wrong_max_identity": ("int32_t lp = (op == OR_MIN) ? INT32_MAX : INT32_MIN;",
                               "int32_t lp = (op == OR_MIN) ? INT32_MAX : 0;"),
    "f32_min_max_transposed": ("float lp = (op == OR_MIN) ? INFINITY : -INFINITY;",
                               "float lp = (op == OR_MIN) ? -INFINITY : INFINITY;"),
    "f32_add_not_accumulated": ("lp += (double)x[i];", "lp = (double)x[i];"),
    "ties_away_from_zero": ("double r = nearbyint(q);", "double r = floor(q + 0.5);"),
    "subnormal_scale_off_by_one": ("v = ldexp((double)m, 1 - bias - f.frac_bits);",
                                   "v = ldexp((double)m, -bias - f.frac_bits);"),
    "f32_store_perturbed": ("float f = (float)v;", "float f = (float)(v * (1.0 + 1e-7));"),
    "select_skips_first": ("if (flags[i] == 1) {", "if (flags[i] == 1 && i > 0) {"),
    "inclusive_stores_before_update": (
        "                lp += (uint32_t)x[i];\n                int32_t v;\n"
        "                memcpy(&v, &lp, 4);\n                y[i] = v;",
        "                int32_t v;\n                memcpy(&v, &lp, 4);\n"
        "                y[i] = v;\n                lp += (uint32_t)x[i];"),
    "inclusive_f32_min_keeps_later": (
        "            float lp = (op == OR_MIN) ? INFINITY : -INFINITY;\n"
        "            for (int64_t i = 0; i < n; ++i) {\n                if (op == OR_MIN)\n"
        "                    lp = (x[i] < lp) ? x[i] : lp;\n                else\n"
        "                    lp = (x[i] > lp) ? x[i] : lp;\n                y[i] = lp;",
        "            float lp = (op == OR_MIN) ? INFINITY : -INFINITY;\n"
        "            for (int64_t i = 0; i < n; ++i) {\n                if (op == OR_MIN)\n"
        "                    lp = (x[i] <= lp) ? x[i] : lp;\n                else\n"
        "                    lp = (x[i] > lp) ? x[i] : lp;\n                y[i] = lp;"),
    "reduce_drops_last": ("            for (int64_t i = 0; i < n; ++i)\n                acc += (uint32_t)x[i];",
                          "            for (int64_t i = 0; i + 1 < n; ++i)\n                acc += (uint32_t)x[i];"),
    "reduce_f32_max_keeps_later": (
        "            r = (op == OR_MIN) ? INFINITY : -INFINITY;\n            for (int64_t i = 0; i < n; ++i)\n"
        "                r = (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);",
        "            r = (op == OR_MIN) ? INFINITY : -INFINITY;\n            for (int64_t i = 0; i < n; ++i)\n"
        "                r = (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] >= r) ? x[i] : r);"),
    "reduce_wrong_min_identity": ("            r = (op == OR_MIN) ? INT64_MAX : INT64_MIN;",
                                  "            r = (op == OR_MIN) ? INT64_MAX : 0;"),
    "rows_prod_seed_zero": ("    if (op == OR_MUL)\n        seed = 1.0;", "    if (op == OR_MUL)\n        seed = 0.0;"),
    "rows_op_min_keeps_later": ("                next = (x < lp) ? x : lp;", "                next = (x <= lp) ? x : lp;"),
    "rows_op_incl_excl_swapped": ("            const double y = inclusive ? next : lp;",
                                  "            const double y = inclusive ? lp : next;"),
    "rows_prod_is_sum": ("                next = lp * x;", "                next = lp + x;"),
    "u32_signed_compare": ("            next = (x[i] < lp) ? x[i] : lp;\n        else\n            next = (x[i] > lp) ? x[i] : lp;\n        y[i] = inclusive ? next : lp;\n        lp = next;\n    }\n}\n\nstatic void scan_u64",
                           "            next = ((int32_t)x[i] < (int32_t)lp) ? x[i] : lp;\n        else\n            next = ((int32_t)x[i] > (int32_t)lp) ? x[i] : lp;\n        y[i] = inclusive ? next : lp;\n        lp = next;\n    }\n}\n\nstatic void scan_u64"),
    "u64_wrong_min_identity": ("    uint64_t lp = (op == OR_MIN) ? UINT64_MAX : 0u;", "    uint64_t lp = (op == OR_MIN) ? INT64_MAX : 0u;"),
    "select_wide_half_copy": ("memcpy((char *)out + j * elem_bytes, (const char *)arr + i * elem_bytes, (size_t)elem_bytes);",
                              "memcpy((char *)out + j * elem_bytes, (const char *)arr + i * elem_bytes, 4);"),
    "rbk_key_compare_bits": ("        return a == b;\n    }\n    uint32_t a, b;", "        return memcmp(&a, &b, 4) == 0;\n    }\n    uint32_t a, b;"),
    "rbk_sum_not_reset": ("            isum = 0;\n            fsum = 0.0;", "            fsum = 0.0;"),
    "rbk_reset_every_element": ("        if (head) {\n            ++r;\n            memcpy((char *)keys_out + 4 * r, (const char *)keys + 4 * i, 4);",
                           "        if (head)\n            ++r;\n        {\n            memcpy((char *)keys_out + 4 * r, (const char *)keys + 4 * i, 4);"),
    "f64_add_wrong_sign": ("            const long double next = lp + (long double)x[i];",
                           "            const long double next = lp - (long double)x[i];"),
}


def _build_mutant(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    src = src.replace(old, new, 1)
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"{name}.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC",
                           "-o", so, c, "-lm"])
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    oracle.lib()  # bind the real one first so argtypes setup is exercised
    with tempfile.TemporaryDirectory() as d:
        so = _build_mutant(name, d)
        monkeypatch.setattr(oracle, "_LIB", so)
        monkeypatch.setattr(oracle, "_SRC", so)  # mtime check: never rebuild over it
        monkeypatch.setattr(oracle, "_lib", None)
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
        monkeypatch.setattr(oracle, "_lib", None)
    assert failed, f"no pin caught the planted mistake {name}"
