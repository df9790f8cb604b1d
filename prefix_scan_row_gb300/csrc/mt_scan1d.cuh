// mt_scan1d.cuh -- configuration and launch of the staged kernel for the
// device-wide 1-D scans, shared by the translation units that instantiate it
// (mt_scan1d.cu: i32, i64, f32; mt_scan1d_ext.cu: u32, u64, f64).
#pragma once

#include "mt_staged.cuh"

namespace mt {

#ifndef MT_SCAN1D_SUB
#define MT_SCAN1D_SUB 3   // sub-tiles per staged super-tile
#endif
#ifndef MT_SCAN1D_SUB8
#define MT_SCAN1D_SUB8 MT_SCAN1D_SUB  // the same for 8-byte types
#endif
#ifndef MT_SCAN1D_ITEMS
#define MT_SCAN1D_ITEMS 4
#endif
#ifndef MT_SCAN1D_THREADS
#define MT_SCAN1D_THREADS 256
#endif
constexpr int kScanItems = MT_SCAN1D_ITEMS;      // 16-byte chunks per thread per tile
constexpr int kScanThreads = MT_SCAN1D_THREADS;  // threads per CTA

#ifndef MT_SCAN1D_F64_RUN
#define MT_SCAN1D_F64_RUN 13  // f64: chunks per thread run (one sub-tile)
#endif

// f64 scans run per-thread runs of consecutive chunks (Staged::tile_lean);
// an odd run length puts the 8 lanes of each shared-memory wavefront on 8
// different 16-byte bank groups.
template <class S>
static constexpr int items_of() {
    return std::is_same<S, double>::value ? MT_SCAN1D_F64_RUN : kScanItems;
}
template <class S>
static constexpr int sub_of() {
    return std::is_same<S, double>::value ? 1 : (sizeof(S) == 8 ? MT_SCAN1D_SUB8 : MT_SCAN1D_SUB);
}

template <class S, class Op>
static cudaError_t launch_scan(const SegArgs &a, const Launch &L) {
    return launch_staged<S, Op, items_of<S>(), sub_of<S>(), kScanThreads>(a, 0, L);
}

template <class S>
static constexpr int64_t tile_elems_of() {
    return Staged<S, OpAdd, items_of<S>(), sub_of<S>(), kScanThreads>::kTE;
}

template <class S>
static cudaError_t launch_op(int op, const SegArgs &a, const Launch &L) {
    switch (op) {
    case 0: return launch_scan<S, OpAdd>(a, L);
    case 1: return launch_scan<S, OpMin>(a, L);
    case 2: return launch_scan<S, OpMax>(a, L);
    default: return cudaErrorInvalidValue;
    }
}

// The segment arguments of one 1-D call.
static SegArgs scan1d_args(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                           bool inclusive, bool aligned_io, const Launch &L) {
    SegArgs a;
    a.in = static_cast<const char *>(arr);
    a.out = static_cast<char *>(out);
    a.nseg = 1;
    a.n = 0;
    a.tpr = 0;
    a.n_dev = n_dev;
    a.counter = reinterpret_cast<unsigned long long *>(scratch);
    a.inclusive = inclusive ? 1 : 0;
    a.aligned_io = aligned_io ? 1 : 0;
    a.lb.recs = scratch + kHeaderSlots;
    a.lb.skip_tile = L.skip_tile;
    a.lb.spin_limit = L.spin_limit;
    a.lb.nrec = 0;        // set by the kernel
    a.out_end = nullptr;  // set by the kernel
    return a;
}

// Reads and clears this translation unit's device error word.
static cudaError_t scan1d_take_error_word(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
