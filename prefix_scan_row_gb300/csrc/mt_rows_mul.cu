// mt_rows_mul.cu -- the row scan with product (the metaltile-std scan.rs
// page, "Multi-op scan variants (prod / max / min)": identity 1.0), f32
// accumulation as for the sum.
#include "mt_rows.cuh"

namespace mt {

cudaError_t rows_launch_mul(const void *in, void *out, int64_t rows, int64_t n, int dtype,
                            const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                            const Launch &L) {
    return rows_launch_op<OpMul>(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
}

cudaError_t rows_mul_take_error(int *code) { return take_error_word(code); }

}  // namespace mt
