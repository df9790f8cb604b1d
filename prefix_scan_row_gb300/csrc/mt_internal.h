// mt_internal.h -- interface between the C-ABI layer (mt_abi.cu) and the
// kernel translation units. Not installed; not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace mt {

constexpr int kMaxDevices = 128;

// A value found once per device (an occupancy, an attribute) and read by any
// host thread: 0 means not known yet; threads that race on the first call
// compute and store the same value.
struct PerDevice {
    std::atomic<int> v[kMaxDevices];
    int get(int dev) const { return v[dev].load(std::memory_order_relaxed); }
    void set(int dev, int x) { v[dev].store(x, std::memory_order_relaxed); }
};

constexpr int kHeaderSlots = 4;              // scratch header: [0] tile counter, rest reserved
constexpr uint32_t kDefaultSpin = 1u << 20;  // look-back polls before a waiter gives up

struct Launch {
    cudaStream_t stream;
    int sm_count;
    int64_t skip_tile;    // look-back test hook (-1: none)
    uint32_t spin_limit;  // look-back poll limit
};

void note_launch();

// Fills L for a launch on `stream` on the current device (its id in *dev):
// SM count, and the look-back test hook's skip tile and poll limit
// (mt_abi.cu). False when the device cannot be queried.
bool make_launch(void *stream, Launch *L, int *dev);

// Whether the kernels can dereference p on device `dev` (mt_abi.cu); `host`
// is set for host memory.
bool ptr_reachable(const void *p, int dev, bool *host);

// ---- launches with programmatic stream serialization ----------------------
// Every kernel of the library is launched so that its CTAs may be scheduled
// while the previous kernel in the stream is still finishing, and starts with
// pdl_prologue(): it first waits until that kernel has completed and its
// writes are visible (stream order is kept exactly), then lets the next
// kernel be scheduled. Back-to-back calls thus lose the launch gap and the
// ramp-up of each grid, not their ordering. Without the launch attribute
// (or after a non-kernel stream operation) the wait returns at once.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_prologue() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <class... KArgs, class... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
#endif

// ---- row-wise scan (mt_rows.cu) -------------------------------------------
struct RowPlan {
    bool staged;             // row longer than one CTA tile: persistent staged kernel
    int items;               // 16-byte chunks per thread
    int64_t tile_elems;      // virtual elements per tile
    int64_t tiles_per_row;   // 1: no look-back (and no workspace)
    int warps;               // single-tile rows: warps per CTA
};
RowPlan rows_plan(int dtype, int64_t n, bool heads_zero);
// op: 0 add, 1 min, 2 max, 3 mul (mt_op)
cudaError_t rows_launch(const void *in, void *out, int64_t rows, int64_t n, int dtype, int op,
                        const RowPlan &p, bool inclusive, bool aligned_io, uint64_t *ws,
                        const Launch &L);
#define MT_ROWS_LAUNCH_DECL(name)                                                                   \
    cudaError_t name(const void *in, void *out, int64_t rows, int64_t n, int dtype, const RowPlan &p, \
                     bool inclusive, bool aligned_io, uint64_t *ws, const Launch &L);
MT_ROWS_LAUNCH_DECL(rows_launch_min)  // mt_rows_minmax.cu
MT_ROWS_LAUNCH_DECL(rows_launch_max)  // mt_rows_minmax.cu
MT_ROWS_LAUNCH_DECL(rows_launch_mul)  // mt_rows_mul.cu
#undef MT_ROWS_LAUNCH_DECL
cudaError_t rows_take_error(int *code);
cudaError_t rows_minmax_take_error(int *code);
cudaError_t rows_mul_take_error(int *code);
int rows_rec_slots();  // 8-byte slots per look-back record of a long row

// ---- device-wide exclusive scan (mt_scan1d.cu) ----------------------------
int64_t scan1d_tile_elems(int dtype);
int scan1d_rec_slots(int dtype);
cudaError_t scan1d_launch(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                          int dtype, int op, bool inclusive, bool aligned_io, const Launch &L);
cudaError_t scan1d_take_error(int *code);
struct SegArgs;
cudaError_t scan1d_launch_ext(const SegArgs &a, int dtype, int op, const Launch &L);  // mt_scan1d_ext.cu
cudaError_t scan1d_ext_take_error(int *code);

// ---- device-wide reduction (mt_reduce.cu) ---------------------------------
int64_t reduce_scratch_slots();  // fixed: header + one partial per CTA
cudaError_t reduce_launch(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                          int dtype, int op, const Launch &L);
cudaError_t reduce_take_error(int *code);

// ---- reduce by key (mt_rbk.cu) ---------------------------------------------
int64_t rbk_tile_elems();
int rbk_rec_slots();
cudaError_t rbk_launch(const void *keys, const void *vals, void *keys_out, void *vals_out, int32_t *num_runs,
                       uint64_t *scratch, const int32_t *n_dev, bool key_float, bool val_float,
                       const Launch &L);
cudaError_t rbk_take_error(int *code);

// ---- select (mt_select.cu) ------------------------------------------------
int64_t select_tile_elems(int elem_bytes);  // 0: the smallest over every element size
int select_rec_slots();
cudaError_t select_launch(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
                          uint64_t *scratch, const int32_t *n_dev, int elem_bytes, const Launch &L);
cudaError_t select_take_error(int *code);

// ---- the no-allocation row scan (mt_noalloc.cu) -----------------------------
cudaError_t noalloc_take_error(int *code);

}  // namespace mt
