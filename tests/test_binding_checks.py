"""The Python binding refuses tensors that the C ABI would misread (strided
views, mismatched dtypes) before it passes any pointer on. Runs on the CPU:
every case is rejected on the host."""
import pytest
import torch

import prefix_scan_row_gb300 as mt


def strided(n, dtype):
    return torch.zeros(2 * n, dtype=dtype)[::2]


I32 = torch.int32


@pytest.mark.parametrize("fn", [mt.mt_exclusive_scan, mt.mt_inclusive_scan])
def test_scans_refuse_strided_views(fn):
    nd = torch.zeros(1, dtype=I32)
    with pytest.raises(ValueError, match="arr must be contiguous"):
        fn(strided(8, I32), torch.zeros(8, dtype=I32), torch.zeros(64, dtype=torch.int64), nd, "add")
    with pytest.raises(ValueError, match="out must be contiguous"):
        fn(torch.zeros(8, dtype=I32), strided(8, I32), torch.zeros(64, dtype=torch.int64), nd, "add")


def test_reduce_select_rbk_refuse_strided_views():
    nd, one = torch.zeros(1, dtype=I32), torch.zeros(1, dtype=I32)
    scr = torch.zeros(64, dtype=torch.int64)
    with pytest.raises(ValueError, match="arr must be contiguous"):
        mt.mt_reduce(strided(8, I32), torch.zeros(1, dtype=I32), scr, nd, "max")
    with pytest.raises(ValueError, match="flags must be contiguous"):
        mt.mt_select(torch.zeros(8, dtype=I32), strided(8, torch.uint8), torch.zeros(8, dtype=I32), one, scr, nd)
    with pytest.raises(ValueError, match="out must be contiguous"):
        mt.mt_select_wide(torch.zeros(8, dtype=torch.int64), torch.zeros(8, dtype=torch.uint8),
                          strided(8, torch.int64), one, scr, nd)
    with pytest.raises(ValueError, match="values_in must be contiguous"):
        mt.mt_reduce_by_key_add(torch.zeros(8, dtype=I32), strided(8, I32), torch.zeros(8, dtype=I32),
                                torch.zeros(8, dtype=I32), one, scr, nd)


def test_dtype_and_shape_mismatches_are_refused():
    nd = torch.zeros(1, dtype=I32)
    with pytest.raises(ValueError):
        mt.mt_exclusive_scan(torch.zeros(8, dtype=I32), torch.zeros(8, dtype=torch.int64),
                             torch.zeros(64, dtype=torch.int64), nd, "add")
    with pytest.raises(ValueError):
        mt.mt_scan_rows(torch.zeros(2, 8), torch.zeros(2, 9), True)
    with pytest.raises(ValueError):
        mt.mt_scan_rows(torch.zeros(4, 8)[:, ::2], torch.zeros(4, 4), True)


def test_select_wide_struct_sizes_must_match():
    """An [n, W] tensor is n structs of W elements; out's structs must have
    arr's size (a 12-byte arr into 8-byte or 16-byte out is refused)."""
    nd, one = torch.zeros(1, dtype=I32), torch.zeros(1, dtype=I32)
    scr = torch.zeros(64, dtype=torch.int64)
    fl = torch.zeros(8, dtype=torch.uint8)
    arr = torch.zeros(8, 3, dtype=I32)
    for out in (torch.zeros(8, dtype=torch.int64), torch.zeros(8, 4, dtype=I32), torch.zeros(8, 6, dtype=torch.int16)[:, :3]):
        with pytest.raises(ValueError):
            mt.mt_select_wide(arr, fl, out, one, scr, nd)
    with pytest.raises(ValueError, match="arr must be contiguous"):
        mt.mt_select_wide(torch.zeros(8, 6, dtype=I32)[:, :3], fl, torch.zeros(8, 3, dtype=I32), one, scr, nd)
