// mt_select.cu -- stream compaction built on an exclusive scan of the flags.
//
// Semantics follow the Quadrants "Algorithms" user guide, section
// "qd.algorithms.select": every arr[i] with flags[i] == 1 lands, in input
// order, in a dense prefix of out; num_out receives the count; the tail of
// out is untouched. The page realises it as a scan of the flags into an
// N-slot index buffer, a scatter pass and a one-thread count pass. Here one
// persistent kernel does all three per tile: it counts the tile's flags,
// gets the tile's output offset from the decoupled look-back, packs the
// selected words in shared memory and writes them out as one contiguous run.
// A value word is only read when one of its four flags is set, so sparse
// flags skip most of the value bytes.
//
// When flags and values are 16-byte aligned, k_select_staged instead brings
// each tile's flags and values into shared memory with two bulk copies and
// publishes the tile's count as soon as they land. Each warp then packs its
// selected words in place at the start of its own range of the tile, walking
// its elements 32 at a time (lane i reads element i of each step, a ballot
// ranks the selected lanes, so the writes are consecutive: no bank
// conflicts). The look-back comes last, then each warp copies its packed run
// out with coalesced stores. k_select serves the other alignments.
#include "mt_lookback.cuh"

namespace mt {

#ifndef MT_SEL_ITEMS
#define MT_SEL_ITEMS 2
#endif
constexpr int kSelItems = MT_SEL_ITEMS;  // flag chunks (16 flags) per thread
constexpr int kSelChunks = kThreads * kSelItems;
constexpr int64_t kSelTE = (int64_t)kSelChunks * 16;  // elements per tile (8192)

struct SelSmem {
    uint32_t warp_tot[kWarps];
    uint32_t prefix;
    unsigned long long tile;
    uint32_t vals[kSelTE];  // the tile's selected words, packed
};

struct SelArgs {
    const void *arr;  // 4-byte (k_select, k_select_staged<uint32_t>) or 8-byte elements
    const uint8_t *flags;
    void *out;
    int32_t *num_out;
    const int32_t *n_dev;
    unsigned long long *counter;
    int aligned;  // flags and arr both 16-byte aligned
    LookBack lb;
};

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int w) {
    return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t keep_low_bytes(uint32_t w, int64_t nbytes) {
    if (nbytes >= 4)
        return w;
    if (nbytes <= 0)
        return 0u;
    return w & ((1u << (8 * (int)nbytes)) - 1u);
}

__global__ void __launch_bounds__(kThreads) k_select(SelArgs a) {
    pdl_prologue();
    __shared__ SelSmem sm;
    const uint32_t *arr = static_cast<const uint32_t *>(a.arr);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t ntiles = (n + kSelTE - 1) / kSelTE;
    for (;;) {
        if (threadIdx.x == 0)
            sm.tile = atomicAdd(a.counter, 1ull);
        __syncthreads();  // also: every thread is done with the previous tile's sm.vals
        const int64_t g = (int64_t)sm.tile;
        if (g >= ntiles)
            break;
        const int64_t t0 = g * kSelTE;

        // Flags: 16 per chunk; bytes at or past n read as 0.
        uint4 f[kSelItems];
#pragma unroll
        for (int j = 0; j < kSelItems; ++j) {
            const int64_t e0 = t0 + (int64_t)(warp * 32 * kSelItems + j * 32 + lane) * 16;
            f[j] = make_uint4(0u, 0u, 0u, 0u);
            if (e0 < n) {
                if (a.aligned) {
                    f[j] = ld_stream(reinterpret_cast<const uint4 *>(a.flags) + e0 / 16);
                } else {
                    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int b = 0; b < 16; ++b)
                        if (e0 + b < n)
                            w[b >> 2] |= (uint32_t)a.flags[e0 + b] << (8 * (b & 3));
                    f[j] = make_uint4(w[0], w[1], w[2], w[3]);
                }
                const int64_t valid = n - e0;
                f[j].x = keep_low_bytes(f[j].x, valid);
                f[j].y = keep_low_bytes(f[j].y, valid - 4);
                f[j].z = keep_low_bytes(f[j].z, valid - 8);
                f[j].w = keep_low_bytes(f[j].w, valid - 12);
            }
        }
        // Values: one 16-byte word group per 4 flags, read only if one is set.
        uint4 v[kSelItems][4];
#pragma unroll
        for (int j = 0; j < kSelItems; ++j) {
            const int64_t e0 = t0 + (int64_t)(warp * 32 * kSelItems + j * 32 + lane) * 16;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t fw = word_of(f[j], w);
                v[j][w] = make_uint4(0u, 0u, 0u, 0u);
                if (fw != 0u) {
                    if (a.aligned) {
                        v[j][w] = ld_stream(reinterpret_cast<const uint4 *>(arr) + (e0 + 4 * w) / 4);
                    } else {
                        uint32_t t[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            if ((fw >> (8 * b)) & 0xffu)
                                t[b] = arr[e0 + 4 * w + b];
                        v[j][w] = make_uint4(t[0], t[1], t[2], t[3]);
                    }
                }
            }
        }

        // Counts per chunk (flags are exactly 0/1, so a popcount counts them).
        uint32_t inc[kSelItems];
#pragma unroll
        for (int j = 0; j < kSelItems; ++j)
            inc[j] = __popc(f[j].x) + __popc(f[j].y) + __popc(f[j].z) + __popc(f[j].w);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
            for (int j = 0; j < kSelItems; ++j) {
                const uint32_t y = __shfl_up_sync(kFull, inc[j], d);
                if (lane >= d)
                    inc[j] += y;
            }
        }
        uint32_t pre[kSelItems];
        uint32_t run = 0u;
#pragma unroll
        for (int j = 0; j < kSelItems; ++j) {
            uint32_t e = __shfl_up_sync(kFull, inc[j], 1);
            if (lane == 0)
                e = 0u;
            pre[j] = run + e;
            run += __shfl_sync(kFull, inc[j], 31);
        }
        if (lane == 0)
            sm.warp_tot[warp] = run;
        __syncthreads();
        uint32_t wpre = 0u, agg = 0u;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t t = sm.warp_tot[w];
            if (w < warp)
                wpre += t;
            agg += t;
        }
        const uint32_t G = tile_prefix<uint32_t, OpAdd>(a.lb, g, 0, agg, &sm.prefix);

        // Pack the selected words of the tile in input order.
#pragma unroll
        for (int j = 0; j < kSelItems; ++j) {
            uint32_t off = wpre + pre[j];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t fw = word_of(f[j], w);
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    if ((fw >> (8 * b)) & 0xffu) {
                        sm.vals[off] = word_of(v[j][w], b);
                        ++off;
                    }
                }
            }
        }
        __syncthreads();
        // One contiguous run per tile: coalesced 4-byte stores.
        uint32_t *dst = static_cast<uint32_t *>(a.out) + G;
        for (uint32_t i = threadIdx.x; i < agg; i += kThreads)
            dst[i] = sm.vals[i];
        if (g == ntiles - 1 && threadIdx.x == 0)
            *a.num_out = (int32_t)(G + agg);
    }
}

// ---- staged variant (16-byte aligned flags and values) ----------------------
// VT: the element type, copied bit for bit (4 or 8 bytes).
template <class VT>
struct SelStagedSmem {
    uint4 flags[kSelChunks];  // 16 flags per chunk
    VT vals[kSelTE];          // the tile's values; each warp packs its selected ones in place
    uint64_t bar_f;           // the flags' copy
    uint64_t bar_v;           // the values' copy
    int64_t tile;
    uint32_t red[kWarps];
    uint32_t prefix;
};

// One staged tile: count and publish the count, pack each warp's selected
// words in place, look back for the tile's output offset, copy the packed
// runs out. FULL: the tile holds kSelTE elements, so no flag or element needs
// a range check. (Looking back before the packing, overlapped with it, was
// measured slower: the look-back then meets more predecessors that have
// only published their counts.)
// Returns false when the values' copy did not complete in time (the caller
// records the error and drains it).
template <bool FULL, class VT>
__device__ __forceinline__ bool select_tile(SelStagedSmem<VT> &sm, const SelArgs &a, int64_t g,
                                            int64_t ntiles, int elems, uint32_t phase) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Count: popcounts of this thread's 16-flag chunks (flags past n are 0).
    uint32_t mine = 0u;
#pragma unroll
    for (int j = 0; j < kSelItems; ++j) {
        const int c = warp * 32 * kSelItems + j * 32 + lane;
        const int valid = elems - c * 16;
        if (FULL || valid > 0) {
            uint4 f = lds128(&sm.flags[c]);
            if (!FULL) {
                f.x = keep_low_bytes(f.x, valid);
                f.y = keep_low_bytes(f.y, valid - 4);
                f.z = keep_low_bytes(f.z, valid - 8);
                f.w = keep_low_bytes(f.w, valid - 12);
            }
            mine += __popc(f.x) + __popc(f.y) + __popc(f.z) + __popc(f.w);
        }
    }
    // The tile's count, published as soon as the flags are in.
    uint32_t wsum = mine;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        wsum += __shfl_xor_sync(kFull, wsum, d);
    if (lane == 0)
        sm.red[warp] = wsum;
    __syncthreads();
    uint32_t agg = 0u, wpre = 0u;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t t = sm.red[w];
        if (w < warp)
            wpre += t;
        agg += t;
    }
    publish_aggregate<uint32_t, OpAdd>(a.lb, g, 0, agg);

    // The values were copied alongside the flags; their copy is the larger one.
    bool ok = true;
    if (threadIdx.x < 32)
        ok = mbar_wait(&sm.bar_v, phase, kCopyWaitLimit);
    if (__syncthreads_or(!ok))
        return false;

    // Pack this warp's selected words in place, in element order. A write
    // goes to a slot at or before every element this warp reads later, and
    // a warp step reads all its lanes before any of them writes.
    const uint8_t *fb = reinterpret_cast<const uint8_t *>(sm.flags);
    const int wstart = warp * 32 * kSelItems * 16;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t cnt = 0u;
#pragma unroll
    for (int step = 0; step < kSelItems * 16; ++step) {
        const int e = wstart + step * 32 + lane;
        const bool sel = (FULL || e < elems) && fb[e] != 0;
        const unsigned bal = __ballot_sync(kFull, sel);
        const VT val = sm.vals[e];
        if (sel)
            sm.vals[wstart + cnt + __popc(bal & lt)] = val;
        cnt += __popc(bal);
    }
    __syncwarp();
    // The tile's output offset (the look-back ends with a block barrier).
    const uint32_t G = lookback_prefix<uint32_t, OpAdd>(a.lb, g, 0, agg, &sm.prefix);
    VT *dst = static_cast<VT *>(a.out) + G + wpre;
    for (uint32_t i = lane; i < cnt; i += 32)
        dst[i] = sm.vals[wstart + i];
    if (g == ntiles - 1 && threadIdx.x == 0)
        *a.num_out = (int32_t)(G + agg);
    return true;
}

template <class VT>
__global__ void __launch_bounds__(kThreads) k_select_staged(SelArgs a) {
    pdl_prologue();
    extern __shared__ __align__(128) unsigned char dsm[];
    SelStagedSmem<VT> &sm = *reinterpret_cast<SelStagedSmem<VT> *>(dsm);
    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t ntiles = (n + kSelTE - 1) / kSelTE;
    if (threadIdx.x == 0) {
        mbar_init(&sm.bar_f, 1);
        mbar_init(&sm.bar_v, 1);
        fence_mbar_init();
    }
    uint32_t phase = 0;
    for (;;) {
        if (threadIdx.x == 0)
            sm.tile = (int64_t)atomicAdd(a.counter, 1ull);
        __syncthreads();  // tile id visible; everyone is done with the last tile
        const int64_t g = sm.tile;
        if (g >= ntiles)
            break;
        const int64_t t0 = g * kSelTE;
        const int elems = (int)((n - t0 < kSelTE) ? n - t0 : kSelTE);
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            const uint32_t fb = (uint32_t)((elems + 15) / 16 * 16);
            const uint32_t vb = (uint32_t)(((int64_t)elems * (int64_t)sizeof(VT) + 15) / 16 * 16);
            mbar_arrive_expect_tx(&sm.bar_f, fb);
            bulk_g2s(&sm.flags[0], a.flags + t0, fb, &sm.bar_f);
            mbar_arrive_expect_tx(&sm.bar_v, vb);
            bulk_g2s(&sm.vals[0], static_cast<const VT *>(a.arr) + t0, vb, &sm.bar_v);
        }
        // Warp 0 waits for the flags; the block barrier passes the
        // completion (and the copied bytes) on to the other warps. The
        // tile's count is published before the values are waited for.
        bool ok = true;
        if (threadIdx.x < 32)
            ok = mbar_wait(&sm.bar_f, phase, kCopyWaitLimit);
        if (__syncthreads_or(!ok))
            ok = false;  // every thread: the flags did not arrive
        else
            ok = (elems == kSelTE) ? select_tile<true, VT>(sm, a, g, ntiles, elems, phase)
                                   : select_tile<false, VT>(sm, a, g, ntiles, elems, phase);
        if (!ok) {  // block-uniform
            if (threadIdx.x == 0) {
                atomicCAS(&g_mt_err, 0, kErrTimeout);
                // drain both copies before leaving
                mbar_wait(&sm.bar_f, phase, kCopyWaitLimit);
                mbar_wait(&sm.bar_v, phase, kCopyWaitLimit);
            }
            return;
        }
        phase ^= 1u;
        fence_proxy_async_smem();  // this thread's shared writes precede the next bulk copies
    }
}

int64_t select_tile_elems() { return kSelTE; }
int select_rec_slots() { return Status<uint32_t>::kSlots; }

template <class VT>
static cudaError_t launch_staged_select(const SelArgs &a, const Launch &L) {
    static PerDevice per_sm;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int bytes = (int)sizeof(SelStagedSmem<VT>);
    int blocks = per_sm.get(dev);
    if (blocks == 0) {
        e = cudaFuncSetAttribute(k_select_staged<VT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(k_select_staged<VT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_select_staged<VT>, kThreads, bytes);
        if (e != cudaSuccess)
            return e;
        blocks = b > 0 ? b : 1;
        per_sm.set(dev, blocks);
    }
    e = launch_pdl(k_select_staged<VT>, (unsigned)(L.sm_count * blocks), kThreads, bytes, L.stream, a);
    note_launch();
    return e;
}

cudaError_t select_launch(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
                          uint64_t *scratch, const int32_t *n_dev, int elem_bytes, bool aligned,
                          const Launch &L) {
    if (aligned || elem_bytes == 8) {  // 8-byte elements: the caller checked the alignment
        SelArgs a;
        a.arr = arr;
        a.flags = flags;
        a.out = out;
        a.num_out = num_out;
        a.n_dev = n_dev;
        a.counter = reinterpret_cast<unsigned long long *>(scratch);
        a.aligned = 1;
        a.lb.recs = scratch + kHeaderSlots;
        a.lb.skip_tile = L.skip_tile;
        a.lb.spin_limit = L.spin_limit;
        return elem_bytes == 8 ? launch_staged_select<uint64_t>(a, L) : launch_staged_select<uint32_t>(a, L);
    }
    static PerDevice per_sm;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int blocks = per_sm.get(dev);
    if (blocks == 0) {
        int b = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_select, kThreads, 0);
        if (err != cudaSuccess)
            return err;
        blocks = b > 0 ? b : 1;
        per_sm.set(dev, blocks);
    }
    SelArgs a;
    a.arr = arr;
    a.flags = flags;
    a.out = out;
    a.num_out = num_out;
    a.n_dev = n_dev;
    a.counter = reinterpret_cast<unsigned long long *>(scratch);
    a.aligned = aligned ? 1 : 0;
    a.lb.recs = scratch + kHeaderSlots;
    a.lb.skip_tile = L.skip_tile;
    a.lb.spin_limit = L.spin_limit;
    const cudaError_t e = launch_pdl(k_select, (unsigned)(L.sm_count * blocks), kThreads, 0, L.stream, a);
    note_launch();
    return e;
}

cudaError_t select_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
