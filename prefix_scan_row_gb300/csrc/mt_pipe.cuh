// mt_pipe.cuh -- persistent, bulk-copy (TMA) pipelined scan over segments.
//
// A segment is a row of a [rows, n] tensor or the whole 1-D array; it is cut
// into tiles of TileScan::kTE virtual elements. Each CTA owns a ring of STAGES
// shared-memory stages. Thread 0 fills a stage with one cp.async.bulk copy of
// a tile (completing on the stage's mbarrier); all threads wait on the
// barrier, copy the tile into registers, and after the block barrier that
// follows those reads thread 0 refills the stage with a later tile -- before
// warp 0 starts the tile's look-back. So while a tile waits for its
// predecessors, STAGES tiles of loads stay in flight.
//
// Tile ids come from an atomic counter (needed with a look-back: a CTA takes
// its ids in increasing order and processes them in that order, so the
// smallest unfinished tile is always some running CTA's current tile), or are
// assigned statically (blockIdx + i * gridDim) when no tile waits on another.
// Thread 0 takes each id one fill ahead to hide the atomic's latency.
//
// Every wait is bounded; a copy that does not complete sets the device error
// word, the CTA waits (bounded) for its other copies in flight, and returns.
#pragma once

#include "mt_tilescan.cuh"

namespace mt {

constexpr uint32_t kCopyWaitLimit = 1u << 26;    // mbarrier polls before giving up
constexpr int64_t kEmptyTile = 1ll << 62;        // tag: tile with no valid element

struct SegArgs {
    const char *in;
    char *out;
    int64_t nseg;                 // number of segments (rows); 1 for a 1-D array
    int64_t n;                    // elements per segment (unused when n_dev is set)
    int64_t tpr;                  // tiles per segment (unused when n_dev is set)
    const int32_t *n_dev;         // 1-D: the live count, read on the device
    unsigned long long *counter;  // dynamic tile ids; nullptr: static assignment
    int inclusive;
    int aligned_io;
    LookBack lb;                  // lb.recs == nullptr: no tile waits on another
};

template <class S, class Op, int ITEMS, int STAGES, int THREADS = kThreads>
struct PipeScan {
    using T = TileScan<S, Op, ITEMS, THREADS>;
    static constexpr int E = T::E;
    struct Smem {
        uint4 stage[STAGES][T::kChunks];
        uint64_t bar[STAGES];
        int64_t tile_of[STAGES];
        typename T::Smem t;
    };
    static constexpr size_t kSmemBytes = sizeof(Smem);

    struct Geo {
        const uint4 *vin;
        S *eout;
        int64_t t0, lo, hi, first;
    };

    __device__ __forceinline__ static void geo(const SegArgs &a, int64_t n, int64_t tpr, int64_t g,
                                               Geo &o) {
        constexpr int64_t s = sizeof(S);
        const int64_t row = g / tpr;
        const int64_t k = g - row * tpr;
        const char *in_row = a.in + row * n * s;
        const int64_t head = (int64_t)(((uintptr_t)in_row & 15u) / s);
        o.vin = reinterpret_cast<const uint4 *>(in_row - head * s);
        o.eout = reinterpret_cast<S *>(a.out + row * n * s) - head;
        o.t0 = k * T::kTE;
        o.lo = head;
        o.hi = head + n;
        o.first = row * tpr;
    }
};

template <class S, class Op, int ITEMS, int STAGES, int THREADS>
__global__ void __launch_bounds__(THREADS) k_scan_pipe(SegArgs a) {
    using P = PipeScan<S, Op, ITEMS, STAGES, THREADS>;
    using T = typename P::T;
    constexpr int E = P::E;
    extern __shared__ __align__(128) unsigned char dsm[];
    typename P::Smem &sm = *reinterpret_cast<typename P::Smem *>(dsm);

    int64_t n, tpr, ntiles;
    if (a.n_dev != nullptr) {
        const int32_t n32 = *a.n_dev;
        n = n32 > 0 ? n32 : 0;
        const int64_t head = (int64_t)(((uintptr_t)a.in & 15u) / sizeof(S));
        tpr = n > 0 ? (head + n + T::kTE - 1) / T::kTE : 1;
        ntiles = n > 0 ? tpr : 0;
    } else {
        n = a.n;
        tpr = a.tpr;
        ntiles = a.nseg * tpr;
    }

    // Producer state, used by thread 0 only.
    int64_t ahead = 0, nstatic = 0;
    auto take = [&]() -> int64_t {
        if (a.counter != nullptr)
            return (int64_t)atomicAdd(a.counter, 1ull);
        return (int64_t)blockIdx.x + (nstatic++) * (int64_t)gridDim.x;
    };
    auto fill = [&](int s, int64_t g) {
        if (g >= ntiles) {
            sm.tile_of[s] = g;
            return;
        }
        typename P::Geo o;
        P::geo(a, n, tpr, g, o);
        const int64_t c0 = o.t0 / E;
        int64_t cend = (o.hi + E - 1) / E;
        if (cend > c0 + T::kChunks)
            cend = c0 + T::kChunks;
        if (cend <= c0) {
            sm.tile_of[s] = g | kEmptyTile;  // a trailing tile past the row's end
            return;
        }
        sm.tile_of[s] = g;
        const uint32_t bytes = (uint32_t)((cend - c0) * 16);
        mbar_arrive_expect_tx(&sm.bar[s], bytes);
        bulk_g2s(&sm.stage[s][0], o.vin + c0, bytes, &sm.bar[s]);
    };
    auto refill = [&](int s) {
        fence_proxy_async_smem();
        const int64_t g2 = ahead;
        if (g2 < ntiles)
            ahead = take();
        fill(s, g2);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s)
            mbar_init(&sm.bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ahead = take();
        for (int s = 0; s < STAGES; ++s) {
            const int64_t g = ahead;
            if (g < ntiles)
                ahead = take();
            fill(s, g);
        }
    }
    __syncthreads();

    uint32_t phases = 0;  // parity of the next completion of each stage's barrier
    for (int64_t k = 0;; ++k) {
        const int s = (int)(k % STAGES);
        const int64_t tag = sm.tile_of[s];
        const int64_t g = tag & ~kEmptyTile;
        if (g >= ntiles)
            break;  // fills are in increasing order: every later stage is past the end too
        if (tag & kEmptyTile) {
            __syncthreads();  // everyone has read tile_of[s] before it is rewritten
            if (threadIdx.x == 0)
                refill(s);
            continue;
        }
        const bool ok = mbar_wait(&sm.bar[s], (phases >> s) & 1u, kCopyWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0)
                atomicCAS(&g_mt_err, 0, kErrTimeout);
            for (int t = 0; t < STAGES; ++t) {  // drain this CTA's copies before leaving
                const int st = (int)((k + t) % STAGES);
                const int64_t tg = sm.tile_of[st];
                if ((tg & kEmptyTile) == 0 && tg < ntiles)
                    mbar_wait(&sm.bar[st], (phases >> st) & 1u, kCopyWaitLimit);
            }
            return;
        }
        phases ^= 1u << s;
        typename P::Geo o;
        P::geo(a, n, tpr, g, o);
        uint4 raw[ITEMS];
        T::load_stage(sm.stage[s], o.t0, o.lo, o.hi, raw);
        auto hook = [&]() {
            if (threadIdx.x == 0)
                refill(s);
        };
        T::scan_store(raw, o.eout, a.aligned_io != 0, o.t0, o.lo, o.hi, a.inclusive != 0, a.lb, g,
                      o.first, sm.t, (int)(k & 1), hook);
    }
}

// The same persistent loop without the shared-memory ring: each tile is read
// straight into registers. A CTA takes a tile id only when it starts loading
// that tile: an id taken earlier but not yet loaded could be the predecessor
// of tiles other CTAs are already scanning, and they would wait for it.
#ifndef MT_DIRECT_MINB
#define MT_DIRECT_MINB 1
#endif
template <class S, class Op, int ITEMS, int THREADS>
__global__ void __launch_bounds__(THREADS, MT_DIRECT_MINB) k_scan_direct(SegArgs a) {
    using P = PipeScan<S, Op, ITEMS, 1, THREADS>;
    using T = typename P::T;
    __shared__ typename T::Smem sm;
    __shared__ int64_t cur_tile;

    int64_t n, tpr, ntiles;
    if (a.n_dev != nullptr) {
        const int32_t n32 = *a.n_dev;
        n = n32 > 0 ? n32 : 0;
        const int64_t head = (int64_t)(((uintptr_t)a.in & 15u) / sizeof(S));
        tpr = n > 0 ? (head + n + T::kTE - 1) / T::kTE : 1;
        ntiles = n > 0 ? tpr : 0;
    } else {
        n = a.n;
        tpr = a.tpr;
        ntiles = a.nseg * tpr;
    }
    for (int64_t k = 0;; ++k) {
        if (threadIdx.x == 0)
            cur_tile = a.counter != nullptr ? (int64_t)atomicAdd(a.counter, 1ull)
                                            : (int64_t)blockIdx.x + k * (int64_t)gridDim.x;
        __syncthreads();  // cur_tile is visible; scan_store has a barrier before its next write
        const int64_t g = cur_tile;
        if (g >= ntiles)
            break;
        typename P::Geo o;
        P::geo(a, n, tpr, g, o);
        if (o.t0 >= o.hi) {  // a trailing tile past the row's end: nobody waits on it
            __syncthreads();
            continue;
        }
        uint4 raw[ITEMS];
        T::load_global(o.vin, o.t0, o.lo, o.hi, raw);
        T::scan_store(raw, o.eout, a.aligned_io != 0, o.t0, o.lo, o.hi, a.inclusive != 0, a.lb, g,
                      o.first, sm, (int)(k & 1), NoHook());
    }
}

template <class S, class Op, int ITEMS, int THREADS>
static cudaError_t launch_direct(const SegArgs &a, int64_t max_ctas, const Launch &L) {
    static int per_sm[128] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_scan_direct<S, Op, ITEMS, THREADS>,
                                                          THREADS, 0);
        if (e != cudaSuccess)
            return e;
        per_sm[dev] = b > 0 ? b : 1;
    }
    int64_t grid = (int64_t)L.sm_count * per_sm[dev];
    if (max_ctas > 0 && grid > max_ctas)
        grid = max_ctas;
    if (grid < 1)
        grid = 1;
    k_scan_direct<S, Op, ITEMS, THREADS><<<(unsigned)grid, THREADS, 0, L.stream>>>(a);
    note_launch();
    return cudaGetLastError();
}

// Host side: persistent grid of (resident CTAs per SM) x SMs, at most max_ctas.
template <class S, class Op, int ITEMS, int STAGES, int THREADS>
static cudaError_t launch_pipe(const SegArgs &a, int64_t max_ctas, const Launch &L) {
    using P = PipeScan<S, Op, ITEMS, STAGES, THREADS>;
    static int per_sm[128] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        e = cudaFuncSetAttribute(k_scan_pipe<S, Op, ITEMS, STAGES, THREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_scan_pipe<S, Op, ITEMS, STAGES, THREADS>,
                                                          THREADS, P::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        per_sm[dev] = b > 0 ? b : 1;
    }
    int64_t grid = (int64_t)L.sm_count * per_sm[dev];
    if (max_ctas > 0 && grid > max_ctas)
        grid = max_ctas;
    if (grid < 1)
        grid = 1;
    k_scan_pipe<S, Op, ITEMS, STAGES, THREADS><<<(unsigned)grid, THREADS, P::kSmemBytes, L.stream>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace mt
