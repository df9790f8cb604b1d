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
#include "mt_tilescan.cuh"

namespace mt {

constexpr int kSelItems = 2;                          // flag chunks (16 flags) per thread
constexpr int kSelChunks = kThreads * kSelItems;
constexpr int64_t kSelTE = (int64_t)kSelChunks * 16;  // elements per tile (8192)

struct SelSmem {
    uint32_t warp_tot[kWarps];
    uint32_t prefix;
    unsigned long long tile;
    uint32_t vals[kSelTE];  // the tile's selected words, packed
};

struct SelArgs {
    const uint32_t *arr;
    const uint8_t *flags;
    uint32_t *out;
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
    __shared__ SelSmem sm;
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
                        v[j][w] = ld_stream(reinterpret_cast<const uint4 *>(a.arr) + (e0 + 4 * w) / 4);
                    } else {
                        uint32_t t[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            if ((fw >> (8 * b)) & 0xffu)
                                t[b] = a.arr[e0 + 4 * w + b];
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
        uint32_t *dst = a.out + G;
        for (uint32_t i = threadIdx.x; i < agg; i += kThreads)
            dst[i] = sm.vals[i];
        if (g == ntiles - 1 && threadIdx.x == 0)
            *a.num_out = (int32_t)(G + agg);
    }
}

int64_t select_tile_elems() { return kSelTE; }
int select_rec_slots() { return Status<uint32_t>::kSlots; }

cudaError_t select_launch(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
                          uint64_t *scratch, const int32_t *n_dev, bool aligned, const Launch &L) {
    static int per_sm = 0;
    if (per_sm == 0) {
        int b = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_select, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        per_sm = b > 0 ? b : 1;
    }
    SelArgs a;
    a.arr = static_cast<const uint32_t *>(arr);
    a.flags = flags;
    a.out = static_cast<uint32_t *>(out);
    a.num_out = num_out;
    a.n_dev = n_dev;
    a.counter = reinterpret_cast<unsigned long long *>(scratch);
    a.aligned = aligned ? 1 : 0;
    a.lb.recs = scratch + kHeaderSlots;
    a.lb.skip_tile = L.skip_tile;
    a.lb.spin_limit = L.spin_limit;
    k_select<<<(unsigned)(L.sm_count * per_sm), kThreads, 0, L.stream>>>(a);
    note_launch();
    return cudaGetLastError();
}

cudaError_t select_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
