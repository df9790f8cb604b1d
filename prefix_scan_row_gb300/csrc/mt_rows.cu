// mt_rows.cu -- row-wise scans along the last axis of a contiguous [rows, n]
// tensor (f32 / bf16 / f16 storage, f32 accumulation): the launch plan, the
// dispatch over the combine operation, and the sum.
//
// Semantics follow the metaltile-std 0.1.0 src/mlx/scan.rs page (module doc
// "Scan benchmark": inclusive out[i] = sum_{j<=i} inp[j], exclusive
// out[i] = sum_{j<i} inp[j] with out[0] = 0, f32 loads and accumulation and
// one cast at the store; section "Multi-op scan variants (prod / max / min)":
// the same scan with product, max or min and identity 1.0, -inf or +inf).
// The page runs one threadgroup per row that walks the row in 1024-element
// chunks with a serial carry; here a row that fits in one tile is one CTA
// (k_scan_rows, mt_tilescan.cuh), and a longer row is split over the
// super-tiles of the persistent staged kernel (mt_staged.cuh) whose carries
// are chained by the decoupled look-back, so every row -- short or 2^24
// long -- is read once and written once.
#include "mt_rows.cuh"

namespace mt {

// Virtual elements per tile of a long row (the same for every operation).
static int64_t long_tile_elems(int dtype) {
    if (dtype == 0)
        return Staged<float, OpAdd, kMultiItems, sub_of<float>(), kMultiThreads>::kTE;
    return Staged<__half, OpAdd, kMultiItems, sub_of<__half>(), kMultiThreads>::kTE;
}

// Single-tile rows: the (warps, chunks per thread) pair that covers the row
// with the least idle chunks, at most 16 warps and 4 chunks per thread (8 for
// f32); ties go to more chunks per thread. Longer rows take the staged path.
RowPlan rows_plan(int dtype, int64_t n, bool heads_zero) {
    const int E = (dtype == 0) ? 4 : 8;
    const int64_t head_max = heads_zero ? 0 : E - 1;
    const int64_t chunks = (head_max + n + E - 1) / E;
    const int max_items = (dtype == 0) ? 8 : 4;
    int best_items = 0, best_warps = 0;
    int64_t best_waste = -1;
    for (int items = 1; items <= max_items; ++items) {
        if (items > 4 && items != 8)
            continue;
        const int64_t warps = (chunks + 32 * items - 1) / (32 * items);
        if (warps > 16)
            continue;
        const int64_t waste = warps * 32 * items - chunks;
        if (best_waste < 0 || waste <= best_waste) {
            best_waste = waste;
            best_items = items;
            best_warps = (int)warps;
        }
    }
    if (best_items > 0)
        return RowPlan{false, best_items, (int64_t)best_warps * 32 * best_items * E, 1, best_warps};
    const int64_t te = long_tile_elems(dtype);
    return RowPlan{true, kMultiItems, te, (head_max + n + te - 1) / te, 0};
}

cudaError_t rows_launch(const void *in, void *out, int64_t rows, int64_t n, int dtype, int op,
                        const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                        const Launch &L) {
    switch (op) {
    case 0: return rows_launch_op<OpAdd>(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
    case 1: return rows_launch_min(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
    case 2: return rows_launch_max(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
    case 3: return rows_launch_mul(in, out, rows, n, dtype, p, inclusive, aligned_io, ws, L);
    default: return cudaErrorInvalidValue;
    }
}

int rows_rec_slots() { return Status<float>::kSlots; }

cudaError_t rows_take_error(int *code) { return take_error_word(code); }

}  // namespace mt
