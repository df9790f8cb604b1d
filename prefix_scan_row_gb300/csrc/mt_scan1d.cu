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
#include "mt_scan1d.cuh"

namespace mt {

int64_t scan1d_tile_elems(int dtype) {
    switch (dtype) {
    case 0: return tile_elems_of<float>();
    case 3: return tile_elems_of<int32_t>();
    case 4: return tile_elems_of<int64_t>();
    case 5: return tile_elems_of<uint32_t>();
    case 6: return tile_elems_of<uint64_t>();
    case 7: return tile_elems_of<double>();
    default: return 0;
    }
}

int scan1d_rec_slots(int dtype) {
    return (dtype == 4 || dtype == 6 || dtype == 7) ? Status<int64_t>::kSlots : Status<int32_t>::kSlots;
}

cudaError_t scan1d_launch(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                          int dtype, int op, bool inclusive, bool aligned_io, const Launch &L) {
    const SegArgs a = scan1d_args(arr, out, scratch, n_dev, inclusive, aligned_io, L);
    switch (dtype) {
    case 0: return launch_op<float>(op, a, L);
    case 3: return launch_op<int32_t>(op, a, L);
    case 4: return launch_op<int64_t>(op, a, L);
    case 5: case 6: case 7: return scan1d_launch_ext(a, dtype, op, L);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t scan1d_take_error(int *code) { return scan1d_take_error_word(code); }

}  // namespace mt
