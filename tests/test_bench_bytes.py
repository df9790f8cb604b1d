"""The algorithmic bytes bench.py divides by: a scan moves 2 s bytes per live
element (one read and one write in its storage width s), over the configured
sizes of the 1-D and row workloads, and a bench step is nine 1-D calls. Each
figure is recomputed here from the workload's own definition, not from
bench.py's helpers."""
import bench
import workloads


def test_live_count_and_capacity():
    assert workloads.SCAN1D_CAPACITY == 2 ** 28
    assert workloads.SCAN1D_LIVE == 2 ** 28 - 12345 == 268_423_111
    assert bench.N_LIVE == workloads.SCAN1D_LIVE


def test_scan_bytes_are_one_read_and_one_write():
    n = 268_423_111
    assert bench.scan_bytes("i32") == 4 * n + 4 * n == 2_147_384_888
    assert bench.scan_bytes("f32") == 2_147_384_888
    assert bench.scan_bytes("i64") == 8 * n + 8 * n == 4_294_769_776
    assert bench.DOM_BYTES == 4_294_769_776


def test_step_is_nine_calls():
    assert bench.CALLS == [(d, op) for d in ("i32", "f32", "i64") for op in ("add", "min", "max")]
    n = 268_423_111
    assert bench.STEP_BYTES == 3 * (8 * n) * 2 + 3 * (16 * n) == 25_768_618_656
    assert bench.STEP_ELEMS == 9 * n


def test_row_call_bytes():
    assert bench.call_bytes(1024, 4096, "f32") == 33_554_432
    assert bench.call_bytes(8192, 8192, "bf16") == 268_435_456
    assert bench.call_bytes(4096, 4099, "f16") == 2 * 2 * 4096 * 4099 == 67_158_016
    assert bench.call_bytes(4, 1 << 24, "f32") == 536_870_912
