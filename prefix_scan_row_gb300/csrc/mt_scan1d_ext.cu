// mt_scan1d_ext.cu -- the device-wide 1-D scans for u32, u64 and f64, the
// dtypes the Quadrants "Algorithms" user guide lists beside i32, i64 and f32
// for its scans (section "qd.algorithms.PrefixSumExecutor"). Unsigned add wraps modulo 2^width and min/max
// compare as unsigned (identities UINT_MAX and 0); f64 follows f32 (identity
// +-inf, earliest element on ties, sums grouped differently from a
// left-to-right loop). Same staged kernel as mt_scan1d.cu.
#include "mt_scan1d.cuh"

namespace mt {

cudaError_t scan1d_launch_ext(const SegArgs &a, int dtype, int op, const Launch &L) {
    switch (dtype) {
    case 5: return launch_op<uint32_t>(op, a, L);
    case 6: return launch_op<uint64_t>(op, a, L);
    case 7: return launch_op<double>(op, a, L);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t scan1d_ext_take_error(int *code) { return scan1d_take_error_word(code); }

}  // namespace mt
