// mt_abi.cu -- the exported C ABI (include/mt_scan.h): argument checks,
// scratch layout and reset, workspace for long rows, launch dispatch.
#include <atomic>
#include <initializer_list>
#include <mutex>

#include "mt_internal.h"
#include "mt_scan.h"

namespace mt {

static std::atomic<uint64_t> g_launches{0};
static std::atomic<int64_t> g_skip_tile{-1};
static std::atomic<uint32_t> g_spin_limit{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Clears the scratch header and the status records a call will use. With a
// device live count, the number of records is worked out on the device from
// *n_dev exactly as the scan kernel does; `num_out` (select only) is set to 0
// so an empty input still reports a count.
__global__ void k_reset(uint64_t *words, int64_t nwords, const int32_t *n_dev, int64_t tile_elems,
                        int elem_size, int head_bytes, int rec_slots, int32_t *num_out) {
    pdl_prologue();
    int64_t total = nwords;
    if (n_dev != nullptr) {
        const int32_t n32 = *n_dev;
        const int64_t n = n32 > 0 ? n32 : 0;
        const int64_t head = head_bytes / elem_size;
        const int64_t ntiles = n > 0 ? (head + n + tile_elems - 1) / tile_elems : 0;
        total = kHeaderSlots + ntiles * rec_slots;
        if (num_out != nullptr && n == 0 && blockIdx.x == 0 && threadIdx.x == 0)
            *num_out = 0;
    }
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride)
        words[i] = 0ull;
}

static int device_sm_count(int *dev_out) {
    static PerDevice cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    if (dev_out)
        *dev_out = dev;
    int c = cache.get(dev);
    if (c == 0) {
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cache.set(dev, c);
    }
    return c;
}

static cudaError_t launch_reset(uint64_t *words, int64_t nwords, const int32_t *n_dev,
                                int64_t tile_elems, int elem_size, int head_bytes, int rec_slots,
                                int32_t *num_out, const Launch &L) {
    int64_t grid;
    if (n_dev == nullptr)
        grid = (nwords + 255) / 256;
    else
        grid = 2 * (int64_t)L.sm_count;  // count unknown on the host: grid-stride
    if (grid < 1)
        grid = 1;
    if (grid > 8 * (int64_t)L.sm_count)
        grid = 8 * (int64_t)L.sm_count;
    const cudaError_t e = launch_pdl(k_reset, (unsigned)grid, 256, 0, L.stream, words, nwords, n_dev,
                                     tile_elems, elem_size, head_bytes, rec_slots, num_out);
    note_launch();
    return e;
}

// A stream-ordered pool per device for the look-back records of long rows.
static std::mutex g_pool_mu;
static cudaMemPool_t g_pool[128] = {};

static cudaError_t device_pool(int dev, cudaMemPool_t *out) {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (g_pool[dev] == nullptr) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaError_t e = cudaMemPoolCreate(&g_pool[dev], &props);
        if (e != cudaSuccess) {
            g_pool[dev] = nullptr;
            return e;
        }
        uint64_t keep = 64ull << 20;  // keep up to 64 MiB cached between calls
        cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep);
    }
    *out = g_pool[dev];
    return cudaSuccess;
}

bool make_launch(void *stream, Launch *L, int *dev) {
    L->stream = static_cast<cudaStream_t>(stream);
    L->sm_count = device_sm_count(dev);
    L->skip_tile = g_skip_tile.load(std::memory_order_relaxed);
    const uint32_t spin = g_spin_limit.load(std::memory_order_relaxed);
    L->spin_limit = spin ? spin : kDefaultSpin;
    return L->sm_count > 0;
}

// The dtypes of the 1-D scans and the reduce.
static bool is_1d_dtype(int dtype) {
    return dtype == MT_F32 || dtype == MT_I32 || dtype == MT_I64 || dtype == MT_U32 || dtype == MT_U64 ||
           dtype == MT_F64;
}

static int elem_size(int dtype) {
    switch (dtype) {
    case MT_F32: case MT_I32: case MT_U32: return 4;
    case MT_BF16: case MT_F16: return 2;
    case MT_I64: case MT_U64: case MT_F64: return 8;
    default: return 0;
    }
}

// Whether the kernels can dereference p: memory of device `dev`, managed
// memory, pinned host memory mapped at the same address, or -- on devices
// that read pageable host memory -- any host address. `host` reports host
// memory.
bool ptr_reachable(const void *p, int dev, bool *host) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        *host = true;
        return false;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
        *host = false;
        return a.device == dev;
    case cudaMemoryTypeManaged:
        *host = false;
        return true;
    case cudaMemoryTypeHost:
        *host = true;
        return a.devicePointer == p;
    default: {  // unregistered host memory
        *host = true;
        static PerDevice pageable;  // 0 unknown, 1 yes, 2 no
        if (dev < 0 || dev >= kMaxDevices)
            return false;
        int known = pageable.get(dev);
        if (known == 0) {
            int v = 0;
            if (cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess)
                v = 0;
            known = v ? 1 : 2;
            pageable.set(dev, known);
        }
        return known == 1;
    }
    }
}

// All of `ps` in device (or managed) memory.
static bool all_device(std::initializer_list<const void *> ps, int dev) {
    for (const void *p : ps) {
        bool host = false;
        if (!ptr_reachable(p, dev, &host) || host)
            return false;
    }
    return true;
}

}  // namespace mt

using namespace mt;

// mt_scan_rows and mt_scan_rows_op share their checks, workspace and kernels.
static int rows_call(const void *inp, void *out, int64_t rows, int64_t n, int dtype, int op,
                     int inclusive, void *stream) {
    if (rows < 0 || n < 0 || op < MT_ADD || op > MT_MUL)
        return MT_ERR_ARG;
    if (dtype != MT_F32 && dtype != MT_BF16 && dtype != MT_F16)
        return MT_ERR_DTYPE;
    if (rows == 0 || n == 0)
        return MT_OK;  // empty input, empty output
    if (inp == nullptr || out == nullptr)
        return MT_ERR_ARG;
    const int64_t s = elem_size(dtype);
    if (((uintptr_t)inp % s) != 0 || ((uintptr_t)out % s) != 0)
        return MT_ERR_ALIGN;
    if (n > INT64_MAX / s / rows)
        return MT_ERR_ARG;
    const bool heads_zero = ((uintptr_t)inp % 16 == 0) && ((n * s) % 16 == 0);
    const bool aligned_io = (((uintptr_t)inp - (uintptr_t)out) % 16) == 0;
    const RowPlan p = rows_plan(dtype, n, heads_zero);
    if (p.tiles_per_row > INT32_MAX / rows)
        return MT_ERR_ARG;  // more CTAs than one launch can take
    Launch L;
    int dev = 0;
    if (!make_launch(stream, &L, &dev))
        return MT_ERR_CUDA;
    bool in_host = false, out_host = false;
    if (!ptr_reachable(inp, dev, &in_host) || !ptr_reachable(out, dev, &out_host))
        return MT_ERR_MEMORY;
    if (p.staged && (in_host || out_host))
        return MT_ERR_MEMORY;  // the long-row kernel bulk-copies from device memory only
    uint64_t *ws = nullptr;
    if (p.tiles_per_row > 1) {
        const int64_t nwords = kHeaderSlots + rows * p.tiles_per_row * rows_rec_slots();
        cudaMemPool_t pool;
        if (device_pool(dev, &pool) != cudaSuccess)
            return MT_ERR_CUDA;
        if (cudaMallocFromPoolAsync((void **)&ws, (size_t)nwords * 8, pool, L.stream) != cudaSuccess)
            return MT_ERR_CUDA;
        if (launch_reset(ws, nwords, nullptr, 0, 1, 0, 1, nullptr, L) != cudaSuccess) {
            cudaFreeAsync(ws, L.stream);
            return MT_ERR_CUDA;
        }
    }
    cudaError_t e = rows_launch(inp, out, rows, n, dtype, op, p, inclusive != 0, aligned_io, ws, L);
    if (ws != nullptr && cudaFreeAsync(ws, L.stream) != cudaSuccess)
        e = cudaErrorUnknown;
    return e == cudaSuccess ? MT_OK : MT_ERR_CUDA;
}

extern "C" int mt_scan_rows(const void *inp, void *out, int64_t rows, int64_t n, int dtype,
                            int inclusive, void *stream) {
    return rows_call(inp, out, rows, n, dtype, MT_ADD, inclusive, stream);
}

extern "C" int mt_scan_rows_op(const void *inp, void *out, int64_t rows, int64_t n, int dtype, int op,
                               int inclusive, void *stream) {
    return rows_call(inp, out, rows, n, dtype, op, inclusive, stream);
}

// The exclusive and inclusive 1-D scans share their checks and kernel.
static int scan1d_call(const void *arr, void *out, void *scratch, const int32_t *n_dev, int dtype,
                       int op, bool inclusive, void *stream) {
    if (!is_1d_dtype(dtype))
        return MT_ERR_DTYPE;
    if (op < MT_ADD || op > MT_MAX)
        return MT_ERR_ARG;
    if (arr == nullptr || out == nullptr || scratch == nullptr || n_dev == nullptr)
        return MT_ERR_ARG;
    if (arr == out && !inclusive)
        return MT_ERR_ALIAS;
    const int s = elem_size(dtype);
    if (((uintptr_t)arr % s) != 0 || ((uintptr_t)out % s) != 0 || ((uintptr_t)scratch % 16) != 0 ||
        ((uintptr_t)n_dev % 4) != 0)
        return MT_ERR_ALIGN;
    Launch L;
    int dev = 0;
    if (!make_launch(stream, &L, &dev))
        return MT_ERR_CUDA;
    if (!all_device({arr, out, scratch, n_dev}, dev))
        return MT_ERR_MEMORY;  // the kernel bulk-copies from, and polls, device memory
    uint64_t *sw = static_cast<uint64_t *>(scratch);
    if (launch_reset(sw, 0, n_dev, scan1d_tile_elems(dtype), s, (int)((uintptr_t)arr & 15u),
                     scan1d_rec_slots(dtype), nullptr, L) != cudaSuccess)
        return MT_ERR_CUDA;
    const bool aligned_io = (((uintptr_t)arr - (uintptr_t)out) % 16) == 0;
    return scan1d_launch(arr, out, sw, n_dev, dtype, op, inclusive, aligned_io, L) == cudaSuccess
               ? MT_OK
               : MT_ERR_CUDA;
}

extern "C" int mt_exclusive_scan(const void *arr, void *out, void *scratch, const int32_t *n_dev,
                                 int dtype, int op, void *stream) {
    return scan1d_call(arr, out, scratch, n_dev, dtype, op, false, stream);
}

extern "C" int mt_inclusive_scan(const void *arr, void *out, void *scratch, const int32_t *n_dev,
                                 int dtype, int op, void *stream) {
    return scan1d_call(arr, out, scratch, n_dev, dtype, op, true, stream);
}

extern "C" int mt_reduce(const void *arr, void *out, void *scratch, const int32_t *n_dev, int dtype,
                         int op, void *stream) {
    if (!is_1d_dtype(dtype))
        return MT_ERR_DTYPE;
    if (op < MT_ADD || op > MT_MAX)
        return MT_ERR_ARG;
    if (arr == nullptr || out == nullptr || scratch == nullptr || n_dev == nullptr)
        return MT_ERR_ARG;
    const int s = elem_size(dtype);
    if (((uintptr_t)arr % s) != 0 || ((uintptr_t)out % s) != 0 || ((uintptr_t)scratch % 8) != 0 ||
        ((uintptr_t)n_dev % 4) != 0)
        return MT_ERR_ALIGN;
    Launch L;
    int dev = 0;
    if (!make_launch(stream, &L, &dev))
        return MT_ERR_CUDA;
    if (!all_device({arr, out, scratch, n_dev}, dev))
        return MT_ERR_MEMORY;
    uint64_t *sw = static_cast<uint64_t *>(scratch);
    if (launch_reset(sw, kHeaderSlots, nullptr, 0, 1, 0, 1, nullptr, L) != cudaSuccess)
        return MT_ERR_CUDA;  // the ticket counter; the partials need no clearing
    return reduce_launch(arr, out, sw, n_dev, dtype, op, L) == cudaSuccess ? MT_OK : MT_ERR_CUDA;
}

// mt_select and mt_select_wide share their checks and kernels.
static int select_call(const void *arr, const uint8_t *flags, void *out, int32_t *num_out, void *scratch,
                       const int32_t *n_dev, int elem_bytes, void *stream) {
    // 4- or 8-byte scalars, or structs of 3 to 64 32-bit words
    if (arr == nullptr || flags == nullptr || out == nullptr || num_out == nullptr ||
        scratch == nullptr || n_dev == nullptr || elem_bytes < 4 || elem_bytes > 256 || elem_bytes % 4 != 0)
        return MT_ERR_ARG;
    if (arr == out)
        return MT_ERR_ALIAS;
    const int align = elem_bytes == 8 ? 8 : 4;  // structs are read as 32-bit words
    if (((uintptr_t)arr % align) != 0 || ((uintptr_t)out % align) != 0 ||
        ((uintptr_t)num_out % 4) != 0 || ((uintptr_t)scratch % 16) != 0 || ((uintptr_t)n_dev % 4) != 0)
        return MT_ERR_ALIGN;
    Launch L;
    int dev = 0;
    if (!make_launch(stream, &L, &dev))
        return MT_ERR_CUDA;
    if (!all_device({arr, flags, out, num_out, scratch, n_dev}, dev))
        return MT_ERR_MEMORY;
    uint64_t *sw = static_cast<uint64_t *>(scratch);
    if (launch_reset(sw, 0, n_dev, select_tile_elems(elem_bytes), 1, 0, select_rec_slots(), num_out, L) !=
        cudaSuccess)
        return MT_ERR_CUDA;
    return select_launch(arr, flags, out, num_out, sw, n_dev, elem_bytes, L) == cudaSuccess
               ? MT_OK
               : MT_ERR_CUDA;
}

extern "C" int mt_select(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
                         void *scratch, const int32_t *n_dev, void *stream) {
    return select_call(arr, flags, out, num_out, scratch, n_dev, 4, stream);
}

extern "C" int mt_select_wide(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
                              void *scratch, const int32_t *n_dev, int elem_bytes, void *stream) {
    return select_call(arr, flags, out, num_out, scratch, n_dev, elem_bytes, stream);
}

extern "C" int mt_reduce_by_key_add(const void *keys_in, const void *values_in, void *keys_out,
                                    void *values_out, int32_t *num_runs, void *scratch,
                                    const int32_t *n_dev, int key_dtype, int value_dtype, void *stream) {
    const auto ok_dtype = [](int d) { return d == MT_I32 || d == MT_U32 || d == MT_F32; };
    if (!ok_dtype(key_dtype) || !ok_dtype(value_dtype))
        return MT_ERR_DTYPE;
    if (keys_in == nullptr || values_in == nullptr || keys_out == nullptr || values_out == nullptr ||
        num_runs == nullptr || scratch == nullptr || n_dev == nullptr)
        return MT_ERR_ARG;
    if (keys_out == keys_in || keys_out == values_in || values_out == keys_in || values_out == values_in)
        return MT_ERR_ALIAS;
    const uintptr_t k = (uintptr_t)keys_in, v = (uintptr_t)values_in;
    if (k % 4 || v % 4 || (uintptr_t)keys_out % 4 || (uintptr_t)values_out % 4 || (uintptr_t)num_runs % 4 ||
        (uintptr_t)scratch % 16 || (uintptr_t)n_dev % 4 || (k % 16) != (v % 16))
        return MT_ERR_ALIGN;  // keys and values are read as aligned 16-byte chunks of the same phase
    Launch L;
    int dev = 0;
    if (!make_launch(stream, &L, &dev))
        return MT_ERR_CUDA;
    if (!all_device({keys_in, values_in, keys_out, values_out, num_runs, scratch, n_dev}, dev))
        return MT_ERR_MEMORY;
    uint64_t *sw = static_cast<uint64_t *>(scratch);
    if (launch_reset(sw, 0, n_dev, rbk_tile_elems(), 4, (int)(k & 15u), rbk_rec_slots(), num_runs, L) !=
        cudaSuccess)
        return MT_ERR_CUDA;
    return rbk_launch(keys_in, values_in, keys_out, values_out, num_runs, sw, n_dev, key_dtype == MT_F32,
                      value_dtype == MT_F32, L) == cudaSuccess
               ? MT_OK
               : MT_ERR_CUDA;
}

extern "C" int64_t mt_scan_scratch_slots(int64_t capacity, int dtype, int kind) {
    if (capacity < 0)
        return -1;
    if (kind == MT_SCRATCH_SCAN) {
        const int64_t te = scan1d_tile_elems(dtype);
        if (te <= 0)
            return -1;
        const int64_t head_max = 16 / elem_size(dtype) - 1;  // a misaligned array start
        const int64_t ntiles = capacity > 0 ? (capacity + head_max + te - 1) / te : 0;
        return kHeaderSlots + ntiles * scan1d_rec_slots(dtype);
    }
    if (kind == MT_SCRATCH_SELECT) {
        const int64_t te = select_tile_elems(0);
        return kHeaderSlots + (capacity + te - 1) / te * select_rec_slots();
    }
    if (kind == MT_SCRATCH_REDUCE_BY_KEY) {
        const int64_t te = rbk_tile_elems();
        const int64_t ntiles = capacity > 0 ? (capacity + 3 + te - 1) / te : 0;  // up to 3 elements of head
        return kHeaderSlots + ntiles * rbk_rec_slots();
    }
    if (kind == MT_SCRATCH_REDUCE)
        return elem_size(dtype) > 0 && dtype != MT_BF16 && dtype != MT_F16 ? reduce_scratch_slots() : -1;
    return -1;
}

extern "C" int64_t mt_scan_rows_scratch_slots(int64_t rows, int64_t n, int dtype) {
    if (rows < 0 || n < 0 || (dtype != MT_F32 && dtype != MT_BF16 && dtype != MT_F16))
        return -1;
    if (rows == 0 || n == 0)
        return 0;
    if (n > INT64_MAX / elem_size(dtype) / rows)
        return -1;
    // the larger of the two plans: a row start on a 16-byte boundary, or not
    int64_t tiles = 1;
    for (const bool heads_zero : {true, false}) {
        const RowPlan p = rows_plan(dtype, n, heads_zero);
        if (p.tiles_per_row > tiles)
            tiles = p.tiles_per_row;
    }
    if (tiles == 1)
        return 0;  // every row fits in one tile: no look-back, no workspace
    if (tiles > (INT64_MAX - kHeaderSlots) / rows_rec_slots() / rows)
        return -1;
    return kHeaderSlots + rows * tiles * rows_rec_slots();
}

extern "C" int mt_scan_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MT_ERR_CUDA;
    int worst = MT_OK;
    cudaError_t (*takers[9])(int *) = {rows_take_error,   rows_minmax_take_error, rows_mul_take_error,
                                       scan1d_take_error, scan1d_ext_take_error,  select_take_error,
                                       rbk_take_error,    noalloc_take_error,     reduce_take_error};
    for (auto take : takers) {
        int code = 0;
        if (take(&code) != cudaSuccess)
            return MT_ERR_CUDA;
        if (code != 0 && worst == MT_OK)
            worst = code;
    }
    return worst;
}

extern "C" uint64_t mt_scan_launches(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int mt_scan_build_checked(void) {
#if defined(MT_CHECKED) && MT_CHECKED
    return 1;
#else
    return 0;
#endif
}

extern "C" const char *mt_scan_strerror(int code) {
    switch (code) {
    case MT_OK: return "ok";
    case MT_ERR_ARG: return "invalid argument";
    case MT_ERR_DTYPE: return "dtype not supported by this call";
    case MT_ERR_ALIAS: return "out aliases the input";
    case MT_ERR_CUDA: return "CUDA error";
    case MT_ERR_LOOKBACK_TIMEOUT: return "look-back wait gave up (results invalid)";
    case MT_ERR_ALIGN: return "pointer misaligned";
    case MT_ERR_TOO_LARGE: return "needs more than the fixed no-allocation scratch (MT_NOALLOC_SCRATCH_BYTES)";
    case MT_ERR_MEMORY: return "a pointer the kernels cannot reach (host memory where device memory is needed)";
    case MT_ERR_BOUNDS: return "a kernel's access fell outside its buffer and was skipped (bounds-checked build)";
    default: return "unknown status";
    }
}

extern "C" int mt_scan_debug_lookback(int64_t skip_publish_tile, uint32_t spin_limit) {
    g_skip_tile.store(skip_publish_tile < 0 ? -1 : skip_publish_tile, std::memory_order_relaxed);
    g_spin_limit.store(spin_limit, std::memory_order_relaxed);
    return MT_OK;
}
