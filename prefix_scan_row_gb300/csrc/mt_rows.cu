// mt_rows.cu -- row-wise sum scan along the last axis of a contiguous
// [rows, n] tensor (f32 / bf16 / f16 storage, f32 accumulation).
//
// Semantics follow the metaltile-std 0.1.0 src/mlx/scan.rs page (module doc
// "Scan benchmark": inclusive out[i] = sum_{j<=i} inp[j], exclusive
// out[i] = sum_{j<i} inp[j] with out[0] = 0, f32 loads and accumulation and
// one cast at the store). The page runs one threadgroup per row that walks
// the row in 1024-element chunks with a serial carry; here a row that fits
// in one tile is one CTA (k_scan_rows, mt_tilescan.cuh), and a longer row is
// split over the super-tiles of the persistent staged kernel (mt_staged.cuh)
// whose carries are chained by the decoupled look-back, so every row --
// short or 2^24 long -- is read once and written once.
#include "mt_staged.cuh"
#include "mt_tilescan.cuh"

namespace mt {

struct RowArgs {
    const char *in;
    char *out;
    int64_t rows;
    int64_t n;
    int inclusive;
    int aligned_io;  // output rows have the input rows' 16-byte phase
};

// One CTA per row; the whole row is one tile of blockDim.x * ITEMS chunks
// (the block size is chosen per row length, up to 16 warps).
// (A minimum-blocks bound, even 1, makes the compiler spend more registers
// here and costs resident CTAs.)
template <class S, int ITEMS>
__global__ void __launch_bounds__(512) k_scan_rows(RowArgs a) {
    pdl_prologue();
    using T = RowTile<S, OpAdd, ITEMS>;
    __shared__ typename T::Smem sm;
    const int64_t row = blockIdx.x;
    if (row >= a.rows)
        return;
    constexpr int64_t s = sizeof(S);
    const char *in_row = a.in + row * a.n * s;
    const int head = (int)(((uintptr_t)in_row & 15u) / s);
    const uint4 *vin = reinterpret_cast<const uint4 *>(in_row - head * s);
    S *eout = reinterpret_cast<S *>(a.out + row * a.n * s) - head;
    const int lo = head, hi = head + (int)a.n;
    if (lo == 0 && hi == (int)blockDim.x * ITEMS * T::E)  // the row fills the tile
        T::template run<true>(vin, eout, a.aligned_io != 0, lo, hi, a.inclusive != 0, sm);
    else
        T::template run<false>(vin, eout, a.aligned_io != 0, lo, hi, a.inclusive != 0, sm);
}

#ifndef MT_ROWS_SUB_WIDE
#define MT_ROWS_SUB_WIDE 3  // sub-tiles per super-tile, 4-byte storage
#endif
#ifndef MT_ROWS_SUB_HALF
#define MT_ROWS_SUB_HALF 2  // 2-byte storage (its f32 prefixes take two planes)
#endif
#ifndef MT_ROWS_THREADS
#define MT_ROWS_THREADS 256
#endif
constexpr int kMultiItems = 4;
constexpr int kMultiThreads = MT_ROWS_THREADS;

template <class S>
static constexpr int sub_of() {
    return sizeof(S) == 2 ? MT_ROWS_SUB_HALF : MT_ROWS_SUB_WIDE;
}

template <class S>
static cudaError_t launch_long(const SegArgs &a, int64_t tiles, const Launch &L) {
    return launch_staged<S, OpAdd, kMultiItems, sub_of<S>(), kMultiThreads>(a, tiles, L);
}

// Virtual elements per tile of a long row.
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

template <class S, int ITEMS>
static cudaError_t launch_one(const RowArgs &a, int64_t grid, int warps, cudaStream_t st) {
    return launch_pdl(k_scan_rows<S, ITEMS>, (unsigned)grid, 32 * warps, 0, st, a);
}

template <class S>
static cudaError_t launch_items(int items, const RowArgs &a, int64_t grid, int warps, cudaStream_t st) {
    switch (items) {
    case 1: return launch_one<S, 1>(a, grid, warps, st);
    case 2: return launch_one<S, 2>(a, grid, warps, st);
    case 3: return launch_one<S, 3>(a, grid, warps, st);
    case 4: return launch_one<S, 4>(a, grid, warps, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t rows_launch(const void *in, void *out, int64_t rows, int64_t n, int dtype,
                        const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                        const Launch &L) {
    if (p.staged) {
        // One super-tile per row needs neither tile ordering nor look-back.
        const bool chained = p.tiles_per_row > 1;
        SegArgs a;
        a.in = static_cast<const char *>(in);
        a.out = static_cast<char *>(out);
        a.nseg = rows;
        a.n = n;
        a.tpr = p.tiles_per_row;
        a.n_dev = nullptr;
        a.counter = chained ? reinterpret_cast<unsigned long long *>(ws) : nullptr;
        a.inclusive = inclusive ? 1 : 0;
        a.aligned_io = aligned_io ? 1 : 0;
        a.lb.recs = chained ? ws + kHeaderSlots : nullptr;
        a.lb.skip_tile = L.skip_tile;
        a.lb.spin_limit = L.spin_limit;
        const int64_t tiles = rows * p.tiles_per_row;
        if (dtype == 0)
            return launch_long<float>(a, tiles, L);
        if (dtype == 1)
            return launch_long<__nv_bfloat16>(a, tiles, L);
        return launch_long<__half>(a, tiles, L);
    }
    RowArgs a;
    a.in = static_cast<const char *>(in);
    a.out = static_cast<char *>(out);
    a.rows = rows;
    a.n = n;
    a.inclusive = inclusive ? 1 : 0;
    a.aligned_io = aligned_io ? 1 : 0;
    cudaError_t e;
    if (dtype == 0)
        e = p.items == 8 ? launch_one<float, 8>(a, rows, p.warps, L.stream)
                         : launch_items<float>(p.items, a, rows, p.warps, L.stream);
    else if (dtype == 1)
        e = launch_items<__nv_bfloat16>(p.items, a, rows, p.warps, L.stream);
    else
        e = launch_items<__half>(p.items, a, rows, p.warps, L.stream);
    note_launch();
    return e;
}

int rows_rec_slots() { return Status<float>::kSlots; }

cudaError_t rows_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
