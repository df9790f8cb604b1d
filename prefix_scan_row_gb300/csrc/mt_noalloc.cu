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
#include <mutex>

#include "mt_internal.h"
#include "mt_scan.h"

namespace mt {

constexpr int64_t kNoAllocSlots = MT_NOALLOC_SCRATCH_BYTES / 8;

// The shared look-back workspace: a tile counter and header, then one 8-byte
// record per tile. Every GPU that loads the library holds it until exit.
// Host code must not use this name as an address: on the host it is only a
// stand-in for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint64_t g_noalloc_scratch[kNoAllocSlots];

// Clears what the next scan reads before writing (the counter and the tile
// records); the previous call leaves its values behind.
__global__ void k_noalloc_clear(int64_t nwords) {
    pdl_prologue();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nwords; i += stride)
        g_noalloc_scratch[i] = 0ull;
}

static std::mutex g_noalloc_mu;
static uint64_t *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached.
static cudaError_t noalloc_scratch(uint64_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_noalloc_ptr[dev] = static_cast<uint64_t *>(p);
    }
    *out = g_noalloc_ptr[dev];
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

    uint64_t *ws = nullptr;
    if (noalloc_scratch(&ws) != cudaSuccess)
        return MT_ERR_CUDA;
    Launch L;
    L.stream = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&L.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MT_ERR_CUDA;
    bool in_host = false, out_host = false;
    if (!ptr_reachable(inp, dev, &in_host) || !ptr_reachable(out, dev, &out_host) ||
        (p.staged && (in_host || out_host)))
        return MT_ERR_MEMORY;  // as mt_scan_rows
    L.skip_tile = -1;
    L.spin_limit = kDefaultSpin;
    if (nwords > 0) {
        int64_t grid = (nwords + 255) / 256;
        if (grid > 1024)
            grid = 1024;
        const cudaError_t e = launch_pdl(k_noalloc_clear, (unsigned)grid, 256, 0, L.stream, nwords);
        note_launch();
        if (e != cudaSuccess)
            return MT_ERR_CUDA;
    } else {
        ws = nullptr;  // rows fit in one tile: no look-back, no workspace
    }
    cudaError_t e = rows_launch(inp, out, rows, n, dtype, MT_ADD, p, inclusive != 0, aligned_io, ws, L);
    return e == cudaSuccess ? MT_OK : MT_ERR_CUDA;
}
