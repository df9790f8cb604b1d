// mt_scan1d.cu -- device-wide exclusive scan (add / min / max over i32, i64
// and f32) with the live count read on the device.
//
// Semantics follow the Quadrants "Algorithms" user guide, section
// "qd.algorithms.exclusive_scan_{add,min,max}": out[i] = op(arr[0:i]), out[0]
// the identity of "Semantics > Common conventions > Identity value". The
// page's realisation is a three-pass scan (tile reduce, scan of partials,
// re-read and scan); here one persistent kernel reads every element once and
// writes it once, chaining tiles with the decoupled look-back. The grid is
// sized from the SM count and occupancy, not from n, so the host never needs
// the live count.
#include "mt_tilescan.cuh"

namespace mt {

constexpr int kScanItems = 4;  // 16 KB of input per tile for every dtype

struct ScanArgs {
    const char *in;
    char *out;
    const int32_t *n_dev;
    unsigned long long *counter;
    int aligned_io;
    LookBack lb;
};

template <class S, class Op>
__global__ void __launch_bounds__(kThreads) k_exclusive_scan(ScanArgs a) {
    using T = TileScan<S, Op, kScanItems>;
    __shared__ typename T::Smem sm;
    constexpr int64_t s = sizeof(S);
    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t head = (int64_t)(((uintptr_t)a.in & 15u) / s);
    const uint4 *vin = reinterpret_cast<const uint4 *>(a.in - head * s);
    S *eout = reinterpret_cast<S *>(a.out) - head;
    const int64_t hi = head + n;
    const int64_t ntiles = n > 0 ? (hi + T::kTE - 1) / T::kTE : 0;
    for (;;) {
        if (threadIdx.x == 0)
            sm.tile = atomicAdd(a.counter, 1ull);
        __syncthreads();
        const int64_t g = (int64_t)sm.tile;
        if (g >= ntiles)
            break;
        // run() contains a block barrier before any thread can come back
        // here and overwrite sm.tile.
        T::run(vin, eout, a.aligned_io != 0, g * T::kTE, head, hi, false, a.lb, g, 0, sm);
    }
}

template <class S>
static constexpr int64_t tile_elems_of() {
    return TileScan<S, OpAdd, kScanItems>::kTE;
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

template <class S, class Op>
static cudaError_t launch(const ScanArgs &a, const Launch &L) {
    static int per_sm = 0;  // resident CTAs per SM for this instance
    if (per_sm == 0) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_exclusive_scan<S, Op>,
                                                                      kThreads, 0);
        if (e != cudaSuccess)
            return e;
        per_sm = b > 0 ? b : 1;
    }
    k_exclusive_scan<S, Op><<<(unsigned)(L.sm_count * per_sm), kThreads, 0, L.stream>>>(a);
    note_launch();
    return cudaGetLastError();
}

template <class S>
static cudaError_t launch_op(int op, const ScanArgs &a, const Launch &L) {
    switch (op) {
    case 0: return launch<S, OpAdd>(a, L);
    case 1: return launch<S, OpMin>(a, L);
    case 2: return launch<S, OpMax>(a, L);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t scan1d_launch(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                          int dtype, int op, bool aligned_io, const Launch &L) {
    ScanArgs a;
    a.in = static_cast<const char *>(arr);
    a.out = static_cast<char *>(out);
    a.n_dev = n_dev;
    a.counter = reinterpret_cast<unsigned long long *>(scratch);
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
