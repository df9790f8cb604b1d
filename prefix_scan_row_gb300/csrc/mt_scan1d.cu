// mt_scan1d.cu -- device-wide exclusive and inclusive scans (add / min / max
// over i32, i64 and f32) with the live count read on the device.
//
// Semantics follow the Quadrants "Algorithms" user guide, section
// "qd.algorithms.exclusive_scan_{add,min,max}": out[i] = op(arr[0:i]), out[0]
// the identity of "Semantics > Common conventions > Identity value". The
// page's realisation is a three-pass scan (tile reduce, scan of partials,
// re-read and scan); here one persistent kernel reads every element once and
// writes it once, chaining super-tiles with the decoupled look-back; each
// super-tile reaches shared memory by one bulk copy (mt_staged.cuh). The grid is
// sized from the SM count and occupancy, not from n, so the host never needs
// the live count.
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

template <class S>
static constexpr int sub_of() {
    return sizeof(S) == 8 ? MT_SCAN1D_SUB8 : MT_SCAN1D_SUB;
}

template <class S, class Op>
static cudaError_t launch_scan(const SegArgs &a, const Launch &L) {
    return launch_staged<S, Op, kScanItems, sub_of<S>(), kScanThreads>(a, 0, L);
}

template <class S>
static constexpr int64_t tile_elems_of() {
    return Staged<S, OpAdd, kScanItems, sub_of<S>(), kScanThreads>::kTE;
}

int64_t scan1d_tile_elems(int dtype) {
    switch (dtype) {
    case 0: return tile_elems_of<float>();
    case 3: return tile_elems_of<int32_t>();
    case 4: return tile_elems_of<int64_t>();
    default: return 0;
    }
}

int scan1d_rec_slots(int dtype) {
    return dtype == 4 ? Status<int64_t>::kSlots : Status<int32_t>::kSlots;
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

cudaError_t scan1d_launch(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                          int dtype, int op, bool inclusive, bool aligned_io, const Launch &L) {
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
    switch (dtype) {
    case 0: return launch_op<float>(op, a, L);
    case 3: return launch_op<int32_t>(op, a, L);
    case 4: return launch_op<int64_t>(op, a, L);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t scan1d_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
