// mt_rows.cuh -- the row-scan kernels and their launch, for one combine
// operation Op (sum, min, max or product). Each operation is instantiated in
// its own translation unit (mt_rows.cu, mt_rows_minmax.cu, mt_rows_mul.cu),
// so the library builds in parallel.
#pragma once

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
// (the block size is chosen per row length, up to 16 warps). Up to 3 chunks
// per thread the kernel fits 40 registers, so 3 blocks of 512 threads (or 6
// of 256) stay resident: short rows then keep more loads in flight per SM.
// With 4 chunks that cap would spill; blocks of at most 256 threads (MAXT)
// ask for 5 resident blocks (48 registers and a few bytes of spill: 80 KB of
// loads in flight per SM instead of 64), and 512-thread blocks for no bound
// (a bound of 1 block of 512 makes the compiler spend more registers than none).
#ifndef MT_ROWS_B4_256
#define MT_ROWS_B4_256 5  // resident 256-thread blocks asked for with 4 chunks per thread (48 registers)
#endif
template <int ITEMS, int MAXT>
constexpr int rows_min_blocks() {
    return MAXT == 256 ? (ITEMS == 4 ? MT_ROWS_B4_256 : 0) : (ITEMS <= 3 ? 3 : 0);
}
template <class S, class Op, int ITEMS, int MAXT>
__global__ void __launch_bounds__(MAXT, (rows_min_blocks<ITEMS, MAXT>())) k_scan_rows(RowArgs a) {
    pdl_prologue();
    using T = RowTile<S, Op, ITEMS>;
    __shared__ typename T::Smem sm;
    const int64_t row = blockIdx.x;
    if (row >= a.rows)
        return;
    constexpr int64_t s = sizeof(S);
    const char *in_row = a.in + row * a.n * s;
    const int head = (int)(((uintptr_t)in_row & 15u) / s);
    const uint4 *vin = reinterpret_cast<const uint4 *>(in_row - head * s);
    S *eout = reinterpret_cast<S *>(a.out + row * a.n * s) - head;
    const char *olo = a.out + row * a.n * s, *ohi = olo + a.n * s;
    const int lo = head, hi = head + (int)a.n;
    if (lo == 0 && hi == (int)blockDim.x * ITEMS * T::E)  // the row fills the tile
        T::template run<true>(vin, eout, a.aligned_io != 0, lo, hi, a.inclusive != 0, sm, olo, ohi);
    else
        T::template run<false>(vin, eout, a.aligned_io != 0, lo, hi, a.inclusive != 0, sm, olo, ohi);
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

template <class S, class Op, int ITEMS>
static cudaError_t launch_one(const RowArgs &a, int64_t grid, int warps, cudaStream_t st) {
    if constexpr (ITEMS == 4) {
        if (warps <= 8)
            return launch_pdl(k_scan_rows<S, Op, ITEMS, 256>, (unsigned)grid, 32 * warps, 0, st, a);
    }
    return launch_pdl(k_scan_rows<S, Op, ITEMS, 512>, (unsigned)grid, 32 * warps, 0, st, a);
}

template <class S, class Op>
static cudaError_t launch_items(int items, const RowArgs &a, int64_t grid, int warps, cudaStream_t st) {
    switch (items) {
    case 1: return launch_one<S, Op, 1>(a, grid, warps, st);
    case 2: return launch_one<S, Op, 2>(a, grid, warps, st);
    case 3: return launch_one<S, Op, 3>(a, grid, warps, st);
    case 4: return launch_one<S, Op, 4>(a, grid, warps, st);
    default: return cudaErrorInvalidValue;
    }
}

// The row scan with combine operation Op, on the plan rows_plan() chose.
template <class Op>
static cudaError_t rows_launch_op(const void *in, void *out, int64_t rows, int64_t n, int dtype,
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
        a.lb.nrec = 0;        // set by the kernel
        a.out_end = nullptr;  // set by the kernel
        const int64_t tiles = rows * p.tiles_per_row;
        if (dtype == 0)
            return launch_staged<float, Op, kMultiItems, sub_of<float>(), kMultiThreads>(a, tiles, L);
        if (dtype == 1)
            return launch_staged<__nv_bfloat16, Op, kMultiItems, sub_of<__nv_bfloat16>(), kMultiThreads>(
                a, tiles, L);
        return launch_staged<__half, Op, kMultiItems, sub_of<__half>(), kMultiThreads>(a, tiles, L);
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
        e = p.items == 8 ? launch_one<float, Op, 8>(a, rows, p.warps, L.stream)
                         : launch_items<float, Op>(p.items, a, rows, p.warps, L.stream);
    else if (dtype == 1)
        e = launch_items<__nv_bfloat16, Op>(p.items, a, rows, p.warps, L.stream);
    else
        e = launch_items<__half, Op>(p.items, a, rows, p.warps, L.stream);
    note_launch();
    return e;
}

// Reads and clears this translation unit's device error word.
static cudaError_t take_error_word(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
