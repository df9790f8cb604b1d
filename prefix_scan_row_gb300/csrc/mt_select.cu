// mt_select.cu -- stream compaction built on an exclusive scan of the flags.
//
// Semantics follow the Quadrants "Algorithms" user guide, section
// "qd.algorithms.select": every arr[i] with flags[i] == 1 lands, in input
// order, in a dense prefix of out; num_out receives the count; the tail of
// out is untouched. The page realises it as a scan of the flags into an
// N-slot index buffer, a scatter pass and a one-thread count pass. Here one
// persistent kernel, k_select_staged, does all three per tile: it brings the
// tile's flags and values into shared memory with two bulk copies, publishes
// the tile's count as soon as the flags land, and gets the tile's output
// offset from the decoupled look-back. Each warp packs its selected words in
// place at the start of its own range of the tile, walking its elements 32
// at a time (lane i reads element i of each step, a ballot ranks the
// selected lanes, so the writes are consecutive: no bank conflicts). The
// look-back comes last, then each warp copies its packed run out with
// coalesced stores. Flags and values may sit at any offset from a 16-byte
// boundary; the copies are widened to the boundaries around the tile.
#include "mt_lookback.cuh"

namespace mt {

// Flag chunks (16 flags each) per thread of a tile: a tile holds 256 x 16 x
// items elements. The staged kernel takes 16384-element tiles for 4-byte
// values and 8192 for 8-byte ones (its shared memory holds a tile's values);
// the struct kernel 8192 (a warp's flags are 32 steps of 32 elements). Each
// tile costs one look-back, whose front moves about 32 tiles per L2 round
// trip, so the elements per tile bound the elements per second.
#ifndef MT_SEL_ITEMS4
#define MT_SEL_ITEMS4 2
#endif
#ifndef MT_SEL_ITEMS8
#define MT_SEL_ITEMS8 2
#endif
constexpr int kSelWordsItems = 2;
#ifndef MT_SEL_GATHER4
#define MT_SEL_GATHER4 0  // sparse tiles of 4-byte values gather (else every tile is staged)
#endif
#ifndef MT_SEL_GATHER8
#define MT_SEL_GATHER8 1  // the same for 8-byte values
#endif
template <class VT>
struct SelShape {
    static constexpr int kItems = sizeof(VT) == 4 ? MT_SEL_ITEMS4 : MT_SEL_ITEMS8;
    static constexpr bool kGather = (sizeof(VT) == 4 ? MT_SEL_GATHER4 : MT_SEL_GATHER8) != 0;
    static constexpr int kChunks = kThreads * kItems;
    static constexpr int64_t kTE = (int64_t)kChunks * 16;  // elements per tile
};
constexpr int kSelWordsChunks = kThreads * kSelWordsItems;
constexpr int64_t kSelWordsTE = (int64_t)kSelWordsChunks * 16;  // elements per struct tile (8192)

struct SelArgs {
    const void *arr;  // 4-byte (k_select_staged<uint32_t>) or 8-byte elements
    const uint8_t *flags;
    void *out;
    int32_t *num_out;
    const int32_t *n_dev;
    unsigned long long *counter;
    LookBack lb;
    const char *out_end;  // one past the call's output (set by the kernel; checked build)
};

__device__ __forceinline__ uint32_t keep_low_bytes(uint32_t w, int64_t nbytes) {
    if (nbytes >= 4)
        return w;
    if (nbytes <= 0)
        return 0u;
    return w & ((1u << (8 * (int)nbytes)) - 1u);
}

// ---- staged kernel (any alignment) -------------------------------------------
// VT: the element type, copied bit for bit (4 or 8 bytes).
//
// The bulk copies start at the 16-byte boundary at or below the tile's first
// flag and first value and end at the boundary at or above its last ones:
// those 16-byte blocks share a page with the tile's own bytes, so the wider
// copy reads nothing that could fault. Flag byte b of the copy holds element
// b - hf and value slot v holds element v - hv, where hf and hv are the
// arrays' offsets from the boundary (the same for every tile, which holds a
// multiple of 16 elements).
template <class VT>
constexpr int kSelValSlots = (int)SelShape<VT>::kTE + 16 / (int)sizeof(VT);
template <class VT>
struct SelStagedSmem {
    uint4 flags[SelShape<VT>::kChunks + 2];  // 16 flags per chunk, hf leading bytes, slack for the last warp
    VT vals[kSelValSlots<VT>];               // the tile's values or the warps' packed runs
    uint64_t bar_f;           // the flags' copy
    uint64_t bar_v;           // the values' copy
    int64_t tile;
    uint32_t red[kWarps];
    uint32_t prefix;
};

// The bytes of a 16-byte flag chunk whose positions lie in [lo, hi).
__device__ __forceinline__ uint4 keep_byte_range(uint4 f, int lo, int hi) {
    f.x = keep_low_bytes(f.x, hi) & ~keep_low_bytes(0xffffffffu, lo);
    f.y = keep_low_bytes(f.y, hi - 4) & ~keep_low_bytes(0xffffffffu, lo - 4);
    f.z = keep_low_bytes(f.z, hi - 8) & ~keep_low_bytes(0xffffffffu, lo - 8);
    f.w = keep_low_bytes(f.w, hi - 12) & ~keep_low_bytes(0xffffffffu, lo - 12);
    return f;
}

// This thread's share of a tile's selected count: popcounts of its 16-flag
// chunks of the copy (warp w owns the flag bytes [512 I w, 512 I (w + 1)) of
// a tile of I chunks per thread; the last warp also the copy's extra chunk
// when hf + elems passes the tile), bytes outside [hf, hf + elems) masked.
// FAST: hf = 0 and a full tile.
template <bool FAST, int ITEMS>
__device__ __forceinline__ uint32_t count_flags(const uint4 *flags, int warp, int lane, int hf, int elems) {
    constexpr int kChunks = kThreads * ITEMS;
    constexpr int kTE = kChunks * 16;
    const int hi = hf + elems;  // one past the copy's last flag byte of the tile
    uint32_t mine = 0u;
#pragma unroll
    for (int j = 0; j < ITEMS; ++j) {
        const int c = warp * 32 * ITEMS + j * 32 + lane;
        if ((FAST || 16 * c < hi) && MT_CHECK_INDEX(c, kChunks + 2)) {
            uint4 f = lds128(&flags[c]);
            if (!FAST)
                f = keep_byte_range(f, hf - 16 * c, hi - 16 * c);
            mine += __popc(f.x) + __popc(f.y) + __popc(f.z) + __popc(f.w);
        }
    }
    if (!FAST && warp == kWarps - 1 && lane == 0 && hi > kTE) {
        const uint4 f = keep_byte_range(lds128(&flags[kChunks]), 0, hi - kTE);
        mine += __popc(f.x) + __popc(f.y) + __popc(f.z) + __popc(f.w);
    }
    return mine;
}

// One staged tile: count and publish the count, gather each warp's selected
// elements into a packed run at the start of its own range of the stage,
// look back for the tile's output offset, copy the packed runs out. Warp w
// owns the flag bytes [1024 w, 1024 (w + 1)) of the copy (the last warp also
// the copy's extra chunk when hf + elems passes the tile) and packs the
// elements they hold. FAST: a full tile with hf = 0 (the flags at a 16-byte
// boundary, the values at any offset hv), so no flag or element needs a range
// check. (Looking back before the packing, overlapped
// with it, was measured slower: the look-back then meets more predecessors
// that have only published their counts.)
//
// The values reach the run one of two ways. A dense tile (more than one
// element in kSelDenseDiv selected) has all its values bulk-copied into the
// stage, and each warp packs its selected ones in place. A sparse tile reads
// only its selected values: every selected lane issues a 4- or 8-byte
// asynchronous copy from HBM straight to its slot of the run, all in flight
// together, so most value sectors are never read. Whether the bulk copy is
// issued is guessed before the flags are counted (the CTA's previous tile:
// density is usually alike across an array) so that the copies of a dense
// tile overlap; a tile guessed sparse that turns out dense issues its copy
// late, and one guessed dense that turns out sparse uses the copied values.
//   v_issued : the values' bulk copy was issued with the flags'
//   vphase   : the parity of the values' barrier phase a copy would complete
//   dense    : set to whether the tile turned out dense (the next guess)
// Returns false when the values' copy did not complete in time (the caller
// records the error; a copy issued here is then drained here).
#ifndef MT_SEL_DENSE_DIV
#define MT_SEL_DENSE_DIV 8  // a tile with more than elems / MT_SEL_DENSE_DIV selected is dense
#endif
constexpr int kSelDenseDiv = MT_SEL_DENSE_DIV;
#ifndef MT_SEL_BATCH
#define MT_SEL_BATCH 8  // packing steps whose loads are issued together
#endif
constexpr int kSelBatch = MT_SEL_BATCH;
#ifndef MT_SEL_CHUNK_BATCH
#define MT_SEL_CHUNK_BATCH 2  // chunk-wise packing steps whose loads are issued together
#endif
constexpr int kSelChunkBatch = MT_SEL_CHUNK_BATCH;
#ifndef MT_SEL_LB_PER_LANE
#define MT_SEL_LB_PER_LANE 2  // predecessors per lane per look-back poll of the staged select
#endif
constexpr int kSelLbPerLane = MT_SEL_LB_PER_LANE;

template <bool FAST, class VT>
__device__ __forceinline__ bool select_tile(SelStagedSmem<VT> &sm, const SelArgs &a, int64_t g,
                                            int64_t ntiles, int elems, int hf_, int hv_, bool v_issued,
                                            uint32_t vphase, bool &dense) {
    using Sh = SelShape<VT>;
    constexpr int kTE = (int)Sh::kTE;
    const int hf = FAST ? 0 : hf_, hv = hv_;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hi = hf + elems;  // one past the copy's last flag byte of the tile
    const bool extra = !FAST && warp == kWarps - 1 && hi > kTE;
    // (the flags' own alignment decides the masking, whatever the values')
    const uint32_t mine = (FAST || (hf == 0 && elems == kTE))
                              ? count_flags<true, Sh::kItems>(sm.flags, warp, lane, 0, kTE)
                              : count_flags<false, Sh::kItems>(sm.flags, warp, lane, hf, elems);
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

    dense = !Sh::kGather || (int64_t)agg * kSelDenseDiv > (int64_t)elems;  // block-uniform
    const bool staged = v_issued || dense;
    if (staged && !v_issued && threadIdx.x == 0) {  // guessed sparse, turned out dense
        const int hvb = hv * (int)sizeof(VT);
        const uint32_t vbytes = (uint32_t)((hvb + (int64_t)elems * (int64_t)sizeof(VT) + 15) / 16 * 16);
        const unsigned char *vsrc = static_cast<const unsigned char *>(a.arr) + g * Sh::kTE * (int64_t)sizeof(VT);
        const uint32_t vb = MT_CHECK_RANGE(&sm.vals[0], vbytes, &sm.vals[0], &sm.vals[kSelValSlots<VT>]) ? vbytes : 0u;
        mbar_arrive_expect_tx(&sm.bar_v, vb);
        if (vb != 0u)
            bulk_g2s(&sm.vals[0], vsrc - hvb, vb, &sm.bar_v);
    }
    if (staged) {
        bool ok = true;
        if (threadIdx.x < 32)
            ok = mbar_wait(&sm.bar_v, vphase, kCopyWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0)
                mbar_wait(&sm.bar_v, vphase, kCopyWaitLimit);  // drain the copy before leaving
            return false;
        }
    }

    const uint8_t *fb = reinterpret_cast<const uint8_t *>(sm.flags);
    const int wstart = warp * 32 * Sh::kItems * 16;
    const int ebase = FAST ? wstart : max(wstart - hf, 0);
    VT *const run = sm.vals + hv + ebase;
    [[maybe_unused]] const int run0 = hv + ebase;  // the run's first slot of sm.vals
    [[maybe_unused]] constexpr int kVals = kSelValSlots<VT>, kFlagBytes = 16 * (Sh::kChunks + 2);
    const unsigned lt = (1u << lane) - 1u;
    uint32_t cnt = 0u;
    if (staged) {
        // Pack this warp's selected words in place, in element order, from
        // the slot of its first element on. A selected element is written at
        // or before its own slot, and every slot read later lies after the
        // slots of the elements read so far; so reads of a batch of steps
        // only need to complete before that batch's writes (the warp
        // barrier), and a batch's loads are all issued together.
        auto batch = [&](int s0, int nsteps) {
            VT v[kSelBatch];
            unsigned bal[kSelBatch];
            bool sel[kSelBatch];
#pragma unroll
            for (int j = 0; j < kSelBatch; ++j) {
                if (j < nsteps) {
                    const int b = wstart + (s0 + j) * 32 + lane;
                    const int e = b - hf;
                    sel[j] = (FAST || (unsigned)e < (unsigned)elems) && MT_CHECK_INDEX(b, kFlagBytes) && fb[b] != 0;
                    bal[j] = __ballot_sync(kFull, sel[j]);
                    v[j] = 0;
                    if (sel[j] && MT_CHECK_INDEX(hv + e, kVals))
                        v[j] = sm.vals[hv + e];
                }
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < kSelBatch; ++j) {
                if (j < nsteps) {
                    if (sel[j] && MT_CHECK_INDEX(run0 + cnt + __popc(bal[j] & lt), kVals))
                        run[cnt + __popc(bal[j] & lt)] = v[j];
                    cnt += __popc(bal[j]);
                }
            }
        };
        static_assert((Sh::kItems * 16) % kSelBatch == 0, "whole batches of steps");
        if constexpr (FAST && sizeof(VT) == 4) {
            // A full tile with its flags at a 16-byte boundary: lane l of
            // step s takes the 4 elements of chunk 32 s + l of the warp's
            // range, as one 4-byte flag word and 16 bytes of values (one
            // aligned chunk, or, with the values hv slots past the boundary,
            // the two aligned chunks around them shifted by hv words; the
            // other words of those chunks belong to neighbouring elements and
            // are dropped, so earlier packing writes that reached them do no
            // harm, while the chunk's own 4 slots lie past every slot an
            // earlier batch wrote). Flags are exactly 0 or 1, so popc(word)
            // is the chunk's count, and the warp's exclusive prefix of those
            // counts (0 to 4) comes from 3 ballots.
            const uint32_t *fw = reinterpret_cast<const uint32_t *>(fb) + wstart / 4;
            const uint4 *vc = reinterpret_cast<const uint4 *>(sm.vals + wstart);
            constexpr int kSteps = Sh::kItems * 4;  // 128 elements per step
            constexpr int kB = kSteps < kSelChunkBatch ? kSteps : kSelChunkBatch;
#pragma unroll
            for (int s0 = 0; s0 < kSteps; s0 += kB) {
                uint32_t f[kB];
                uint4 v[kB];
#pragma unroll
                for (int j = 0; j < kB; ++j) {
                    f[j] = MT_CHECK_INDEX(wstart / 4 + (s0 + j) * 32 + lane, kFlagBytes / 4) ? fw[(s0 + j) * 32 + lane] : 0u;
                    v[j] = make_uint4(0u, 0u, 0u, 0u);
                    const int c = (s0 + j) * 32 + lane;
                    if (f[j] != 0u && MT_CHECK_INDEX(wstart / 4 + c, kVals / 4)) {
                        const uint4 p = lds128(&vc[c]);
                        if (hv == 0) {  // block-uniform
                            v[j] = p;
                        } else {
                            const uint4 q = MT_CHECK_INDEX(wstart / 4 + c + 1, kVals / 4) ? lds128(&vc[c + 1])
                                                                                        : make_uint4(0u, 0u, 0u, 0u);
                            v[j] = hv == 1 ? make_uint4(p.y, p.z, p.w, q.x)
                                           : (hv == 2 ? make_uint4(p.z, p.w, q.x, q.y) : make_uint4(p.w, q.x, q.y, q.z));
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int j = 0; j < kB; ++j) {
                    const uint32_t k = __popc(f[j]);
                    const unsigned b1 = __ballot_sync(kFull, k & 1u), b2 = __ballot_sync(kFull, k & 2u),
                                   b4 = __ballot_sync(kFull, k & 4u);
                    uint32_t o = cnt + __popc(b1 & lt) + 2u * __popc(b2 & lt) + 4u * __popc(b4 & lt);
                    if (!MT_CHECK_RANGE(run + o, 4u * __popc(f[j]), &sm.vals[0], &sm.vals[kVals]))
                        f[j] = 0u;  // checked build: skip this word's stores
                    if (f[j] & 0x000000ffu)
                        run[o++] = v[j].x;
                    if (f[j] & 0x0000ff00u)
                        run[o++] = v[j].y;
                    if (f[j] & 0x00ff0000u)
                        run[o++] = v[j].z;
                    if (f[j] & 0xff000000u)
                        run[o] = v[j].w;
                    cnt += __popc(b1) + 2u * __popc(b2) + 4u * __popc(b4);
                }
                __syncwarp();  // this batch's writes before the next batch's reads
            }
        } else {
#pragma unroll 1
            for (int s0 = 0; s0 < Sh::kItems * 16; s0 += kSelBatch)
                batch(s0, kSelBatch);
            if (extra)  // warp-uniform
                batch(Sh::kItems * 16, 1);
        }
    } else {
        // Gather each selected value from HBM into its slot of the run; the
        // copies complete while warp 0 looks back.
        const VT *src = static_cast<const VT *>(a.arr) + g * Sh::kTE;
        auto step = [&](int s) {
            const int b = wstart + s * 32 + lane;
            const int e = b - hf;
            const bool sel = (FAST || (unsigned)e < (unsigned)elems) && MT_CHECK_INDEX(b, kFlagBytes) && fb[b] != 0;
            const unsigned bal = __ballot_sync(kFull, sel);
            if (sel && MT_CHECK_INDEX(run0 + cnt + __popc(bal & lt), kVals))
                cp_async_small<(int)sizeof(VT)>(run + cnt + __popc(bal & lt), src + e);
            cnt += __popc(bal);
        };
#pragma unroll
        for (int s = 0; s < Sh::kItems * 16; ++s)
            step(s);
        if (extra)  // warp-uniform
            step(Sh::kItems * 16);
    }
    // The tile's output offset (the look-back ends with a block barrier).
    const uint32_t G = lookback_prefix<uint32_t, OpAdd, kSelLbPerLane>(a.lb, g, 0, agg, &sm.prefix);
    if (!staged)
        cp_async_wait_all();
    __syncwarp();
    VT *dst = static_cast<VT *>(a.out) + G + wpre;
    for (uint32_t i = lane; i < cnt; i += 32)
        if (MT_CHECK_INDEX(run0 + i, kVals) && MT_CHECK_RANGE(dst + i, sizeof(VT), a.out, a.out_end))
            dst[i] = run[i];
    if (g == ntiles - 1 && threadIdx.x == 0)
        *a.num_out = (int32_t)(G + agg);
    return true;
}

// Resident blocks per SM that the shared memory allows (the bound keeps the
// registers within that): 5 for 8192 4-byte values, 2 for 16384; 3 for
// 8192 8-byte values.
template <class VT>
constexpr int sel_staged_minb() {
    return (int)((227u * 1024u) / (sizeof(SelStagedSmem<VT>) + 1024u));
}
template <class VT>
__global__ void __launch_bounds__(kThreads, sel_staged_minb<VT>()) k_select_staged(SelArgs a) {
    pdl_prologue();
    constexpr int64_t kSelTE = SelShape<VT>::kTE;
    extern __shared__ __align__(128) unsigned char dsm[];
    SelStagedSmem<VT> &sm = *reinterpret_cast<SelStagedSmem<VT> *>(dsm);
    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t ntiles = (n + kSelTE - 1) / kSelTE;
    a.lb.nrec = ntiles;
    a.out_end = static_cast<const char *>(a.out) + n * (int64_t)sizeof(VT);
    // Offsets from the 16-byte boundary below (arr is aligned to its element size).
    const int hf = (int)(reinterpret_cast<uintptr_t>(a.flags) & 15u);
    const int hvb = (int)(reinterpret_cast<uintptr_t>(a.arr) & 15u);
    const int hv = hvb / (int)sizeof(VT);
    if (threadIdx.x == 0) {
        mbar_init(&sm.bar_f, 1);
        mbar_init(&sm.bar_v, 1);
        fence_mbar_init();
    }
    uint32_t fphase = 0, vphase = 0;
    bool guess_dense = true;  // whether to copy the values along with the flags (always, without gathering)
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
            uint32_t fbytes = (uint32_t)((hf + elems + 15) / 16 * 16);
            if (!MT_CHECK_RANGE(&sm.flags[0], fbytes, &sm.flags[0], &sm.flags[SelShape<VT>::kChunks + 2]))
                fbytes = 0u;  // checked build: no copy (the phase completes with no bytes)
            mbar_arrive_expect_tx(&sm.bar_f, fbytes);
            if (fbytes != 0u)
                bulk_g2s(&sm.flags[0], a.flags + t0 - hf, fbytes, &sm.bar_f);
            if (guess_dense) {
                uint32_t vbytes = (uint32_t)((hvb + (int64_t)elems * (int64_t)sizeof(VT) + 15) / 16 * 16);
                const unsigned char *vsrc = static_cast<const unsigned char *>(a.arr) + t0 * (int64_t)sizeof(VT);
                if (!MT_CHECK_RANGE(&sm.vals[0], vbytes, &sm.vals[0], &sm.vals[kSelValSlots<VT>]))
                    vbytes = 0u;
                mbar_arrive_expect_tx(&sm.bar_v, vbytes);
                if (vbytes != 0u)
                    bulk_g2s(&sm.vals[0], vsrc - hvb, vbytes, &sm.bar_v);
            }
        }
        // Warp 0 waits for the flags; the block barrier passes the
        // completion (and the copied bytes) on to the other warps. The
        // tile's count is published before the values are waited for.
        bool ok = true;
        if (threadIdx.x < 32)
            ok = mbar_wait(&sm.bar_f, fphase, kCopyWaitLimit);
        bool dense = guess_dense;
        if (__syncthreads_or(!ok)) {  // every thread: the flags did not arrive
            if (threadIdx.x == 0) {
                mbar_wait(&sm.bar_f, fphase, kCopyWaitLimit);  // drain the copies before leaving
                if (guess_dense)
                    mbar_wait(&sm.bar_v, vphase, kCopyWaitLimit);
            }
            ok = false;
        } else {
            ok = (elems == kSelTE && hf == 0)  // a full tile with aligned flags (the values at any offset)
                     ? select_tile<true, VT>(sm, a, g, ntiles, elems, hf, hv, guess_dense, vphase, dense)
                     : select_tile<false, VT>(sm, a, g, ntiles, elems, hf, hv, guess_dense, vphase, dense);
        }
        if (!ok) {  // block-uniform
            if (threadIdx.x == 0)
                atomicCAS(&g_mt_err, 0, kErrTimeout);
            return;
        }
        fphase ^= 1u;
        if (guess_dense || dense)  // a values copy completed
            vphase ^= 1u;
        guess_dense = dense;
        fence_proxy_async_smem();  // this thread's shared writes precede the next bulk copies
    }
}

// ---- struct elements ----------------------------------------------------------
// Elements of W 32-bit words (W >= 3: 12 to 256 bytes, 4-byte aligned), as
// the page's select takes struct element types and copies them field by
// field. A tile of 8192 elements would need up to 2 MB of shared memory for
// its values, so only the flags are staged: the tile's count is published,
// the look-back gives its output offset, and then each warp copies its
// selected elements straight from arr to out. Each warp first takes the
// ballots of its 32 steps of 32 elements (lane s keeps step s's ballot and
// the count of selected elements before it); then lane k copies the warp's
// k-th selected element, E elements per lane per round, all their words in
// flight together. WT: W known at compile time (0: at run time).
struct SelWordsSmem {
    uint4 flags[kSelWordsChunks + 2];  // as in SelStagedSmem
    uint64_t bar_f;
    int64_t tile;
    uint32_t red[kWarps];
    uint32_t prefix;
};

struct SelWords {
    int words;  // W
    int vec;    // W a multiple of 4 and arr, out 16-byte aligned: copy 16-byte vectors
};

// Selected elements per lane per round, and resident CTAs per SM asked of
// the compiler, per struct size (measured at p = 0.5 and 0.01 on 2^28
// structs: 12 bytes best at 3 and 5, 16 bytes at 3 and 4; no spills).
__host__ __device__ constexpr int sel_words_e(int wt) { return wt == 3 || wt == 4 ? 3 : (wt == 6 ? 2 : 1); }
#ifndef MT_SEL_WORDS_MINB
__host__ __device__ constexpr int sel_words_minb(int wt) { return wt == 3 ? 5 : 4; }
#else
__host__ __device__ constexpr int sel_words_minb(int) { return MT_SEL_WORDS_MINB; }
#endif

template <bool FAST, int WT>
__device__ __forceinline__ void select_words_tile(SelWordsSmem &sm, const SelArgs &a, int W_rt, int vec,
                                                  int64_t g, int64_t ntiles, int elems, int hf_) {
    constexpr int kTE = (int)kSelWordsTE;
    const int W = WT != 0 ? WT : W_rt;
    const int hf = FAST ? 0 : hf_;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t mine = count_flags<FAST, kSelWordsItems>(sm.flags, warp, lane, hf, elems);
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
    // The tile's output offset (the look-back ends with a block barrier).
    const uint32_t G = lookback_prefix<uint32_t, OpAdd>(a.lb, g, 0, agg, &sm.prefix);

    const uint8_t *fb = reinterpret_cast<const uint8_t *>(sm.flags);
    const uint32_t *src = static_cast<const uint32_t *>(a.arr);
    uint32_t *dst = static_cast<uint32_t *>(a.out);
    const int wstart = warp * 32 * kSelWordsItems * 16;
    const int64_t t0 = g * kSelWordsTE;
    static_assert(kSelWordsItems * 16 == 32, "a warp's flag bytes are 32 steps of 32");
    // The ballots of the warp's 32 steps of 32 elements: lane s keeps step
    // s's ballot and the number of selected elements in the steps before s.
    unsigned my_bal = 0u;
#pragma unroll 8
    for (int st = 0; st < 32; ++st) {
        const int bb = wstart + st * 32 + lane;
        const int e = bb - hf;
        const bool sel = (FAST || (unsigned)e < (unsigned)elems) && MT_CHECK_INDEX(bb, 16 * (kSelWordsChunks + 2)) &&
                         fb[bb] != 0;
        const unsigned bal = __ballot_sync(kFull, sel);
        if (lane == st)
            my_bal = bal;
    }
    uint32_t my_before = __popc(my_bal);
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, my_before, d);
        if (lane >= d)
            my_before += y;
    }
    const uint32_t warp_cnt = __shfl_sync(kFull, my_before, 31);
    my_before -= __popc(my_bal);  // exclusive
    const int64_t ibase = (t0 + wstart - hf) * (int64_t)W;  // word 0 of the warp's element 0
    const uint32_t obase = G + wpre;
    // Lane k of a round copies the warp's k-th selected element: a 5-step
    // shuffle search over the step counts finds its step, a 5-step popcount
    // search in that step's ballot its lane. Every lane has work at any
    // density, the search is paid once per element (not per word), and E
    // elements' W words are all loaded before any is stored. The words of one
    // element are adjacent and the elements of a round nearly so, so the
    // round's loads and stores touch few sectors beyond the ones they need.
#ifdef MT_SEL_WORDS_E
    constexpr int E = MT_SEL_WORDS_E;
#else
    constexpr int E = sel_words_e(WT);  // selected elements per lane per round
#endif
    constexpr int C = WT != 0 ? WT : 8;  // words in flight per element (run time W: chunks of 8)
    for (uint32_t k0 = 0; k0 < warp_cnt; k0 += 32 * E) {
        int el[E];  // the warp-local element of this lane's x-th selected element, -1 past the count
#pragma unroll
        for (int x = 0; x < E; ++x) {
            const uint32_t k = k0 + 32 * x + lane;
            int st = 0;  // the step holding selected element k: the last with my_before <= k
#pragma unroll
            for (int d = 16; d > 0; d >>= 1)
                if (__shfl_sync(kFull, my_before, st + d) <= k)
                    st += d;
            const unsigned bal = __shfl_sync(kFull, my_bal, st);
            int rk = (int)(k - __shfl_sync(kFull, my_before, st));  // its rank within the step
            int pos = 0;  // the rk-th set bit of bal
#pragma unroll
            for (int w = 16; w > 0; w >>= 1) {
                const int c = __popc((bal >> pos) & ((1u << w) - 1u));
                if (rk >= c) {
                    rk -= c;
                    pos += w;
                }
            }
            el[x] = k < warp_cnt ? st * 32 + pos : -1;
        }
        if (WT == 0 && vec) {  // launch-uniform: 16-byte loads and stores (W at run time: 8 words and up)
            const uint4 *src4 = reinterpret_cast<const uint4 *>(src);
            uint4 *dst4 = reinterpret_cast<uint4 *>(dst);
            const int W4 = W / 4;
            constexpr int C4 = C / 4 > 0 ? C / 4 : 1;  // (only W at run time takes this branch: C = 8)
#pragma unroll 1
            for (int w0 = 0; w0 < W4; w0 += C4) {
                uint4 v[E][C4];
#pragma unroll
                for (int x = 0; x < E; ++x)
#pragma unroll
                    for (int w = 0; w < C4; ++w)
                        if (el[x] >= 0 && (WT != 0 || w0 + w < W4))
                            v[x][w] = __ldg(src4 + ibase / 4 + (int64_t)el[x] * W4 + w0 + w);
#pragma unroll
                for (int x = 0; x < E; ++x) {
                    const int64_t o = (int64_t)(obase + k0 + 32 * x + lane) * W4 + w0;
#pragma unroll
                    for (int w = 0; w < C4; ++w)
                        if (el[x] >= 0 && (WT != 0 || w0 + w < W4) && MT_CHECK_RANGE(dst4 + o + w, 16, a.out, a.out_end))
                            dst4[o + w] = v[x][w];
                }
            }
            continue;
        }
#pragma unroll 1
        for (int w0 = 0; w0 < W; w0 += C) {
            uint32_t v[E][C];
#pragma unroll
            for (int x = 0; x < E; ++x)
#pragma unroll
                for (int w = 0; w < C; ++w)
                    if (el[x] >= 0 && (WT != 0 || w0 + w < W))
                        v[x][w] = __ldg(src + ibase + (int64_t)el[x] * W + w0 + w);
#pragma unroll
            for (int x = 0; x < E; ++x) {
                const int64_t o = (int64_t)(obase + k0 + 32 * x + lane) * W + w0;
#pragma unroll
                for (int w = 0; w < C; ++w)
                    if (el[x] >= 0 && (WT != 0 || w0 + w < W) && MT_CHECK_RANGE(dst + o + w, 4, a.out, a.out_end))
                        dst[o + w] = v[x][w];
            }
        }
    }
    // The copy's extra chunk (last warp only, when hf + elems passes the
    // tile): at most 15 elements, one per lane.
    if (!FAST && warp == kWarps - 1 && hf + elems > kTE) {
        const int bb = wstart + 1024 + lane;
        const int e = bb - hf;
        const bool sel = (unsigned)e < (unsigned)elems && MT_CHECK_INDEX(bb, 16 * (kSelWordsChunks + 2)) && fb[bb] != 0;
        const unsigned bal = __ballot_sync(kFull, sel);
        if (sel) {
            const int64_t in = ibase + (int64_t)(1024 + lane) * W;
            const int64_t o = (int64_t)(obase + warp_cnt + __popc(bal & ((1u << lane) - 1u))) * W;
            for (int w = 0; w < W; ++w)
                if (MT_CHECK_RANGE(dst + o + w, 4, a.out, a.out_end))
                    dst[o + w] = __ldg(src + in + w);
        }
    }
    if (g == ntiles - 1 && threadIdx.x == 0)
        *a.num_out = (int32_t)(G + agg);
}

template <int WT>
__global__ void __launch_bounds__(kThreads, sel_words_minb(WT)) k_select_words(SelArgs a, SelWords sw) {
    pdl_prologue();
    __shared__ __align__(128) SelWordsSmem sm;
    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t ntiles = (n + kSelWordsTE - 1) / kSelWordsTE;
    a.lb.nrec = ntiles;
    a.out_end = static_cast<const char *>(a.out) + n * (int64_t)sw.words * 4;
    const int hf = (int)(reinterpret_cast<uintptr_t>(a.flags) & 15u);
    if (threadIdx.x == 0) {
        mbar_init(&sm.bar_f, 1);
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
        const int64_t t0 = g * kSelWordsTE;
        const int elems = (int)((n - t0 < kSelWordsTE) ? n - t0 : kSelWordsTE);
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();
            uint32_t fbytes = (uint32_t)((hf + elems + 15) / 16 * 16);
            if (!MT_CHECK_RANGE(&sm.flags[0], fbytes, &sm.flags[0], &sm.flags[kSelWordsChunks + 2]))
                fbytes = 0u;  // checked build: no copy (the phase completes with no bytes)
            mbar_arrive_expect_tx(&sm.bar_f, fbytes);
            if (fbytes != 0u)
                bulk_g2s(&sm.flags[0], a.flags + t0 - hf, fbytes, &sm.bar_f);
        }
        bool ok = true;
        if (threadIdx.x < 32)
            ok = mbar_wait(&sm.bar_f, phase, kCopyWaitLimit);
        if (__syncthreads_or(!ok)) {  // block-uniform: the flags did not arrive
            if (threadIdx.x == 0) {
                atomicCAS(&g_mt_err, 0, kErrTimeout);
                mbar_wait(&sm.bar_f, phase, kCopyWaitLimit);  // drain the copy before leaving
            }
            return;
        }
        if (elems == kSelWordsTE && hf == 0)
            select_words_tile<true, WT>(sm, a, sw.words, sw.vec, g, ntiles, elems, hf);
        else
            select_words_tile<false, WT>(sm, a, sw.words, sw.vec, g, ntiles, elems, hf);
        phase ^= 1u;
        fence_proxy_async_smem();  // this thread's shared reads precede the next bulk copy
    }
}

template <int WT>
static cudaError_t launch_words_select(const SelArgs &a, const SelWords &sw, const Launch &L) {
    static PerDevice per_sm;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int blocks = per_sm.get(dev);
    if (blocks == 0) {
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_select_words<WT>, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        blocks = b > 0 ? b : 1;
        per_sm.set(dev, blocks);
    }
    e = launch_pdl(k_select_words<WT>, (unsigned)(L.sm_count * blocks), kThreads, 0, L.stream, a, sw);
    note_launch();
    return e;
}

int64_t select_tile_elems(int elem_bytes) {
    if (elem_bytes == 4)
        return SelShape<uint32_t>::kTE;
    if (elem_bytes == 8)
        return SelShape<uint64_t>::kTE;
    if (elem_bytes > 8)
        return kSelWordsTE;
    // any element size: the smallest tile (the most status records)
    int64_t t = SelShape<uint32_t>::kTE < SelShape<uint64_t>::kTE ? SelShape<uint32_t>::kTE : SelShape<uint64_t>::kTE;
    return t < kSelWordsTE ? t : kSelWordsTE;
}
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
                          uint64_t *scratch, const int32_t *n_dev, int elem_bytes, const Launch &L) {
    SelArgs a;
    a.arr = arr;
    a.flags = flags;
    a.out = out;
    a.num_out = num_out;
    a.n_dev = n_dev;
    a.counter = reinterpret_cast<unsigned long long *>(scratch);
    a.lb.recs = scratch + kHeaderSlots;
    a.lb.skip_tile = L.skip_tile;
    a.lb.spin_limit = L.spin_limit;
    a.lb.nrec = 0;        // set by the kernel
    a.out_end = nullptr;  // set by the kernel
    if (elem_bytes == 4)
        return launch_staged_select<uint32_t>(a, L);
    if (elem_bytes == 8)
        return launch_staged_select<uint64_t>(a, L);
    SelWords sw;
    sw.words = elem_bytes / 4;
    sw.vec = (elem_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(arr) % 16 == 0 &&
              reinterpret_cast<uintptr_t>(out) % 16 == 0) ? 1 : 0;
    switch (sw.words) {  // the struct sizes the page names: 3, 4 and 6 words; others at run time
    case 3:
        return launch_words_select<3>(a, sw, L);
    case 4:
        return launch_words_select<4>(a, sw, L);
    case 6:
        return launch_words_select<6>(a, sw, L);
    default:
        return launch_words_select<0>(a, sw, L);
    }
}

cudaError_t select_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
