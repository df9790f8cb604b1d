// mt_noalloc.cu -- mt_scan_rows_noalloc: the row scan for callers that may
// not allocate device memory.
//
// Some programs cannot let a library allocate: their device memory is all
// reserved up front by another allocator, or they call the scan from a loop
// where an allocation could take a driver lock or wait on the device, or
// their host forbids device allocations after start-up. mt_scan_rows needs a
// small look-back workspace for rows longer than one tile and takes it from
// a memory pool; this variant uses one fixed array that lives in the library
// instead, so nothing is allocated. The pages describe no such variant.
#include <cuda.h>  // CUcontext / CUresult types only; the calls come through the runtime

#include <mutex>

#include "mt_internal.h"
#include "mt_scan.h"
#include "mt_tile.cuh"

namespace mt {

constexpr int64_t kNoAllocSlots = MT_NOALLOC_SCRATCH_BYTES / 8;

// The shared look-back workspace: the header slots (the tile counter first),
// then one status record per tile of rows_rec_slots() 8-byte slots (one
// 128-byte line). Every GPU that loads the library holds it until exit.
// Host code must not use this name as an address: on the host it is only a
// stand-in for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocSlots];

// Clears what the next scan reads before writing (the counter and the tile
// records); the previous call leaves its values behind.
__global__ void k_noalloc_clear(int64_t nwords) {
    pdl_prologue();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nwords; i += stride)
        if (MT_CHECK_INDEX(i, kNoAllocSlots))
            g_noalloc_scratch[i] = 0ull;
}

// The process-unique id of the context current on this thread, or 0 when
// there is none (or the driver does not offer the calls). The driver calls
// are fetched through the runtime, so the library does not link libcuda.
static unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static std::once_flag once;
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        (void)cudaGetLastError();
    });
    if (get_current == nullptr || get_id == nullptr)
        return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the array in the current context, cached per device with
// the id of the context it was found in. A device reset, or a context of the
// caller's own made current, gives a new context whose copy of the array may
// sit elsewhere: the address is then looked up again (with that context
// current), never reused from another context.
struct NoAllocEntry {
    unsigned long long ctx;
    uint64_t *ptr;
};
static std::mutex g_noalloc_mu;
static NoAllocEntry g_noalloc_cache[kMaxDevices] = {};

static cudaError_t noalloc_scratch(int dev, uint64_t **out) {
    unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocEntry &e = g_noalloc_cache[dev];
    if (ctx == 0 || e.ptr == nullptr || e.ctx != ctx) {
        void *p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess)
            return err;
        // the lookup makes the device's context current if none was
        e.ctx = ctx != 0 ? ctx : current_context_id();
        e.ptr = static_cast<uint64_t *>(p);
    }
    *out = e.ptr;
    return cudaSuccess;
}

}  // namespace mt

using namespace mt;

extern "C" int mt_scan_rows_noalloc(const void *inp, void *out, int64_t rows, int64_t n, int dtype,
                                    int inclusive, void *stream) {
    if (rows < 0 || n < 0)
        return MT_ERR_ARG;
    if (dtype != MT_F32 && dtype != MT_BF16 && dtype != MT_F16)
        return MT_ERR_DTYPE;
    if (rows == 0 || n == 0)
        return MT_OK;
    if (inp == nullptr || out == nullptr)
        return MT_ERR_ARG;
    const int64_t s = (dtype == MT_F32) ? 4 : 2;
    if (((uintptr_t)inp % s) != 0 || ((uintptr_t)out % s) != 0)
        return MT_ERR_ALIGN;
    if (n > INT64_MAX / s / rows)
        return MT_ERR_ARG;
    const bool heads_zero = ((uintptr_t)inp % 16 == 0) && ((n * s) % 16 == 0);
    const bool aligned_io = (((uintptr_t)inp - (uintptr_t)out) % 16) == 0;
    const RowPlan p = rows_plan(dtype, n, heads_zero);
    if (p.tiles_per_row > INT32_MAX / rows)
        return MT_ERR_ARG;
    const int64_t nwords =
        (p.tiles_per_row > 1) ? kHeaderSlots + rows * p.tiles_per_row * rows_rec_slots() : 0;
    if (nwords > kNoAllocSlots)
        return MT_ERR_TOO_LARGE;

    Launch L;
    int dev = 0;
    if (!make_launch(stream, &L, &dev))
        return MT_ERR_CUDA;
    bool in_host = false, out_host = false;
    if (!ptr_reachable(inp, dev, &in_host) || !ptr_reachable(out, dev, &out_host) ||
        (p.staged && (in_host || out_host)))
        return MT_ERR_MEMORY;  // as mt_scan_rows
    uint64_t *ws = nullptr;
    if (nwords > 0) {  // rows longer than one tile: look-back records in the fixed array
        if (noalloc_scratch(dev, &ws) != cudaSuccess)
            return MT_ERR_CUDA;
        int64_t grid = (nwords + 255) / 256;
        if (grid > 1024)
            grid = 1024;
        const cudaError_t e = launch_pdl(k_noalloc_clear, (unsigned)grid, 256, 0, L.stream, nwords);
        note_launch();
        if (e != cudaSuccess)
            return MT_ERR_CUDA;
    }
    const cudaError_t e = rows_launch(inp, out, rows, n, dtype, MT_ADD, p, inclusive != 0, aligned_io, ws, L);
    return e == cudaSuccess ? MT_OK : MT_ERR_CUDA;
}

namespace mt {
// Reads and clears this translation unit's device error word (set only by
// the bounds-checked build's checks of the clear kernel).
cudaError_t noalloc_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}
}  // namespace mt
