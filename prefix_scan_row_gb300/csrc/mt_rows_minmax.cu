// mt_rows_minmax.cu -- the row scans with max and min (the metaltile-std
// scan.rs page, "Multi-op scan variants (prod / max / min)": identity -inf
// and +inf). min/max keep the earlier operand on ties, so every grouping
// gives the bits of a left-to-right fold.
#include "mt_rows.cuh"

namespace mt {

cudaError_t rows_launch_min(const void *in, void *out, int64_t rows, int64_t n, int dtype,
                            const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                            const Launch &L) {
    return rows_launch_op<OpMin>(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
}

cudaError_t rows_launch_max(const void *in, void *out, int64_t rows, int64_t n, int dtype,
                            const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                            const Launch &L) {
    return rows_launch_op<OpMax>(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
}

cudaError_t rows_minmax_take_error(int *code) { return take_error_word(code); }

}  // namespace mt
