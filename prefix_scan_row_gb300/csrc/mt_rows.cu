// mt_rows.cu -- row-wise sum scan along the last axis of a contiguous
// [rows, n] tensor (f32 / bf16 / f16 storage, f32 accumulation).
//
// Semantics follow the metaltile-std 0.1.0 src/mlx/scan.rs page (module doc
// "Scan benchmark": inclusive out[i] = sum_{j<=i} inp[j], exclusive
// out[i] = sum_{j<i} inp[j] with out[0] = 0, f32 loads and accumulation and
// one cast at the store). The page runs one threadgroup per row that walks
// the row in 1024-element chunks with a serial carry; here a row that fits
// in one tile is one CTA, and a longer row is split over several CTAs whose
// carries are chained by the decoupled look-back, so every row -- short or
// 2^24 long -- is read once and written once.
#include "mt_tilescan.cuh"

namespace mt {

struct RowArgs {
    const char *in;
    char *out;
    int64_t rows;
    int64_t n;
    int64_t tpr;                  // tiles per row
    int inclusive;
    int aligned_io;               // output rows have the input rows' 16-byte phase
    unsigned long long *counter;  // dynamic tile ids (multi-tile rows only)
    LookBack lb;
};

template <class S, int ITEMS>
__global__ void __launch_bounds__(kThreads) k_scan_rows(RowArgs a) {
    using T = TileScan<S, OpAdd, ITEMS>;
    __shared__ typename T::Smem sm;
    int64_t g;
    if (a.lb.recs == nullptr) {
        g = blockIdx.x;  // one tile per row: no ordering needed
    } else {
        // Tile ids in the order CTAs start, so every tile a CTA waits on has
        // already been taken by a running CTA.
        if (threadIdx.x == 0)
            sm.tile = atomicAdd(a.counter, 1ull);
        __syncthreads();
        g = (int64_t)sm.tile;
    }
    const int64_t row = g / a.tpr;
    const int64_t k = g - row * a.tpr;
    if (row >= a.rows)
        return;
    constexpr int64_t s = sizeof(S);
    const char *in_row = a.in + row * a.n * s;
    const int64_t head = (int64_t)(((uintptr_t)in_row & 15u) / s);
    const uint4 *vin = reinterpret_cast<const uint4 *>(in_row - head * s);
    S *eout = reinterpret_cast<S *>(a.out + row * a.n * s) - head;
    const int64_t t0 = k * T::kTE;
    const int64_t hi = head + a.n;
    if (t0 >= hi)
        return;  // an empty trailing tile: nothing to do, and nobody waits on it
    T::run(vin, eout, a.aligned_io != 0, t0, head, hi, a.inclusive != 0, a.lb, g, row * a.tpr, sm);
}

// Chunks per thread tried for rows that fit in one tile; longer rows use
// kMultiItems per tile (16 KB of input per tile).
constexpr int kMultiItems = 4;

RowPlan rows_plan(int dtype, int64_t n, bool heads_zero) {
    const int E = (dtype == 0) ? 4 : 8;
    const int64_t head_max = heads_zero ? 0 : E - 1;
    const int max_items = (dtype == 0) ? 8 : 4;
    for (int items = 1; items <= max_items; items *= 2) {
        const int64_t te = (int64_t)kThreads * items * E;
        if (head_max + n <= te)
            return RowPlan{items, te, 1};
    }
    const int64_t te = (int64_t)kThreads * kMultiItems * E;
    return RowPlan{kMultiItems, te, (head_max + n + te - 1) / te};
}

template <class S, int ITEMS>
static void launch_one(const RowArgs &a, int64_t grid, cudaStream_t st) {
    k_scan_rows<S, ITEMS><<<(unsigned)grid, kThreads, 0, st>>>(a);
}

template <class S>
static void launch_items(int items, const RowArgs &a, int64_t grid, cudaStream_t st) {
    switch (items) {
    case 1: launch_one<S, 1>(a, grid, st); break;
    case 2: launch_one<S, 2>(a, grid, st); break;
    case 4: launch_one<S, 4>(a, grid, st); break;
    default: break;
    }
}

cudaError_t rows_launch(const void *in, void *out, int64_t rows, int64_t n, int dtype,
                        const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                        const Launch &L) {
    RowArgs a;
    a.in = static_cast<const char *>(in);
    a.out = static_cast<char *>(out);
    a.rows = rows;
    a.n = n;
    a.tpr = p.tiles_per_row;
    a.inclusive = inclusive ? 1 : 0;
    a.aligned_io = aligned_io ? 1 : 0;
    a.counter = reinterpret_cast<unsigned long long *>(ws);
    a.lb.recs = (p.tiles_per_row > 1) ? ws + kHeaderSlots : nullptr;
    a.lb.skip_tile = L.skip_tile;
    a.lb.spin_limit = L.spin_limit;
    const int64_t grid = rows * p.tiles_per_row;
    if (dtype == 0) {
        if (p.items == 8)
            launch_one<float, 8>(a, grid, L.stream);
        else
            launch_items<float>(p.items, a, grid, L.stream);
    } else if (dtype == 1) {
        launch_items<__nv_bfloat16>(p.items, a, grid, L.stream);
    } else {
        launch_items<__half>(p.items, a, grid, L.stream);
    }
    note_launch();
    return cudaGetLastError();
}

cudaError_t rows_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
