// mt_lookback.cuh -- single-pass decoupled look-back across the tiles of one
// segment (a row, or the whole 1-D array).
//
// Each tile owns a status record in device scratch. After its local reduce a
// tile publishes its aggregate (flag kAgg); warp 0 then walks back over its
// predecessors 32 at a time (one lane per predecessor), folding aggregates
// until it meets a predecessor that has published an inclusive prefix
// (kIncl); it then publishes its own inclusive prefix. The first tile of a
// segment publishes its aggregate as inclusive at once. Tile ids come from an
// atomic counter in launch order, so every tile waited on belongs to a CTA
// that is already running: the wait always ends.
//
// Every wait is bounded: after `spin_limit` polls (or once another tile has
// recorded an error) the waiter records MT_ERR_LOOKBACK_TIMEOUT in the
// device error word, publishes what it has so later tiles are not held, and
// carries on. Results are then invalid but the kernel ends and the context
// stays usable.
#pragma once

#include "mt_tile.cuh"

namespace mt {

#ifndef MT_REC_SLOTS
#define MT_REC_SLOTS 16  // 8-byte slots per record: one 128-byte line each, so the
                         // records near the look-back front spread over L2 slices
#endif
#if MT_REC_SLOTS < 2
#error "a record needs at least two 8-byte slots for 8-byte values"
#endif

// Tile status records.
template <class Acc, bool kPacked = (sizeof(Acc) == 4)> struct Status;

// 4-byte values: one 8-byte word, flag in the high half and value bits in the
// low half. A 64-bit store or load is single-copy atomic, and the value needs
// no other data, so relaxed gpu-scope order is enough.
template <class Acc> struct Status<Acc, true> {
    static constexpr int kSlots = MT_REC_SLOTS;
    __device__ __forceinline__ static void publish(uint64_t *rec, uint32_t flag, Acc v) {
        st_relaxed_u64(rec, ((uint64_t)flag << 32) | bits32<Acc>(v));
    }
    __device__ __forceinline__ static void read(const uint64_t *rec, uint32_t &flag, Acc &v) {
        const uint64_t w = ld_relaxed_u64(rec);
        flag = (uint32_t)(w >> 32);
        v = from32<Acc>((uint32_t)w);
    }
};

// 8-byte values: two words, each [flag:32 | one 32-bit half of the value]
// (low half first). Every word is written by one single-copy-atomic 64-bit
// store and carries the flag of the state it belongs to, so a reader that
// loads both words (two independent loads: one round trip) and finds the
// same flag in both has both halves of that state's value. A reader that
// finds two different flags caught the record between the two stores of an
// update and sees it as empty, which only makes it poll again. States only
// move forward (empty, aggregate, inclusive), so no fence is needed.
template <class Acc> struct Status<Acc, false> {
    static constexpr int kSlots = MT_REC_SLOTS;
    __device__ __forceinline__ static void publish(uint64_t *rec, uint32_t flag, Acc v) {
        const uint64_t u = bits64<Acc>(v);
        const uint64_t f = (uint64_t)flag << 32;
        st_relaxed_u64(rec, f | (u & 0xffffffffull));
        st_relaxed_u64(rec + 1, f | (u >> 32));
    }
    __device__ __forceinline__ static void read(const uint64_t *rec, uint32_t &flag, Acc &v) {
        const uint64_t w0 = ld_relaxed_u64(rec);
        const uint64_t w1 = ld_relaxed_u64(rec + 1);
        const uint32_t f0 = (uint32_t)(w0 >> 32), f1 = (uint32_t)(w1 >> 32);
        flag = (f0 == f1) ? f0 : kEmpty;
        v = from64<Acc>((w1 << 32) | (w0 & 0xffffffffull));
    }
};

struct LookBack {
    uint64_t *recs;      // tile records; nullptr when every segment is one tile
    int64_t skip_tile;   // test hook: this tile never publishes (-1: none)
    uint32_t spin_limit; // polls before a waiter gives up
    int64_t nrec;        // records of the call (set by the kernel; bounds every publish in a checked build)
};

// Publishes `v` with `flag` in tile `t`'s record (the checked build first
// checks that t is a record of the call).
template <class Acc>
__device__ __forceinline__ void publish_record(const LookBack &lb, int64_t t, uint32_t flag, Acc v) {
    if (MT_CHECK_INDEX(t, lb.nrec))
        Status<Acc>::publish(lb.recs + t * Status<Acc>::kSlots, flag, v);
}

#ifndef MT_LB_PER_LANE
#define MT_LB_PER_LANE 1
#endif
// Predecessors read by each lane per poll: the window is 32 * kLbPerLane tiles.
// The inclusive-prefix front advances by at most one window per L2 round trip,
// so the window bounds the scan's throughput at window x tile bytes / latency.
constexpr int kLbPerLane = MT_LB_PER_LANE;

// Called by all 32 lanes of warp 0. Returns the exclusive prefix of `tile`
// (the combine of every earlier tile of the segment [first, tile)).
// Lane l reads tiles pos - l*K - i, i = 0..K-1 (i = 0 newest), so lanes hold
// consecutive groups and a higher lane always holds older tiles.
template <class Acc, class Op, int K = kLbPerLane>
__device__ __forceinline__ Acc warp_lookback(const uint64_t *recs, int64_t tile, int64_t first,
                                             uint32_t spin_limit) {
    using St = Status<Acc>;
    const int lane = threadIdx.x & 31;
    const Acc ident = Op::template identity<Acc>();
    Acc excl = ident;
    int64_t pos = tile - 1;  // the newest predecessor not yet folded
    uint32_t polls = 0;
    for (;;) {
        uint32_t f[K];
        Acc v[K];
#pragma unroll
        for (int i = 0; i < K; ++i) {
            const int64_t t = pos - (int64_t)lane * K - i;
            f[i] = kIncl;  // before the segment start: an inclusive identity
            v[i] = ident;
            if (t >= first)
                St::read(recs + t * St::kSlots, f[i], v[i]);
        }
        // Nearest inclusive predecessor within this lane's group (K: none),
        // and whether a tile this lane must fold is still empty.
        int inc_i = K;
#pragma unroll
        for (int i = K - 1; i >= 0; --i)
            if (f[i] == kIncl)
                inc_i = i;
        bool blocked = false;
#pragma unroll
        for (int i = 0; i < K; ++i)
            if (i <= inc_i && f[i] == kEmpty)
                blocked = true;
        const unsigned incl = __ballot_sync(kFull, inc_i < K);
        const unsigned low = incl & (0u - incl);                  // lane of the nearest inclusive
        const unsigned need = incl ? (low | (low - 1u)) : kFull;  // lanes that must be folded
        if (__ballot_sync(kFull, blocked) & need) {
            ++polls;
            bool give_up = polls >= spin_limit;
            if (!give_up && (polls & 63u) == 0)
                give_up = ld_relaxed_i32(&g_mt_err) != 0;
            if (__any_sync(kFull, give_up)) {
                if (lane == 0)
                    atomicCAS(&g_mt_err, 0, kErrTimeout);
                return excl;
            }
            if (polls > 8)
                __nanosleep(polls < 64 ? 64 : 256);
            continue;
        }
        // Fold this lane's group, oldest first, stopping at its inclusive one.
        Acc c = ident;
        if ((need >> lane) & 1u) {
#pragma unroll
            for (int i = K - 1; i >= 0; --i)
                if (i <= inc_i)
                    c = Op::apply(c, v[i]);
        }
        // Ordered fold across lanes: a higher lane holds older tiles (left).
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const Acc o = __shfl_down_sync(kFull, c, d);
            if (lane + d < 32)
                c = Op::apply(o, c);
        }
        c = __shfl_sync(kFull, c, 0);
        excl = Op::apply(c, excl);
        if (incl)
            return excl;
        pos -= 32 * K;
    }
}

// Thread 0 publishes this tile's aggregate: as the inclusive prefix for the
// first tile of a segment, as an aggregate otherwise.
template <class Acc, class Op>
__device__ __forceinline__ void publish_aggregate(const LookBack &lb, int64_t tile, int64_t first,
                                                  Acc agg) {
    using St = Status<Acc>;
    if (lb.recs == nullptr || threadIdx.x != 0 || tile == lb.skip_tile)
        return;
    publish_record<Acc>(lb, tile, tile == first ? kIncl : kAgg, agg);
}

// Block-wide, after publish_aggregate: warp 0 looks back, thread 0 publishes
// the inclusive prefix; every thread gets the tile's exclusive prefix.
// `tile` and `first` are block-uniform; `agg` is needed in thread 0 only.
// (The whole block reading one group of 32 predecessors per warp, 256 per
// round trip, was measured slower for every kernel: the polling traffic
// costs more than the round trips it saves.)
template <class Acc, class Op, int K = kLbPerLane>
__device__ __forceinline__ Acc lookback_prefix(const LookBack &lb, int64_t tile, int64_t first,
                                               Acc agg, Acc *sm_prefix) {
    using St = Status<Acc>;
    const Acc ident = Op::template identity<Acc>();
    if (lb.recs == nullptr || tile == first)
        return ident;
    if (threadIdx.x < 32) {
        const Acc ex = warp_lookback<Acc, Op, K>(lb.recs, tile, first, lb.spin_limit);
        if (threadIdx.x == 0) {
            if (tile != lb.skip_tile)
                publish_record<Acc>(lb, tile, kIncl, Op::apply(ex, agg));
            *sm_prefix = ex;
        }
    }
    __syncthreads();
    return *sm_prefix;
}

// Both steps at once: publish the aggregate, look back, publish the inclusive
// prefix, and return the tile's exclusive prefix to every thread.
template <class Acc, class Op>
__device__ __forceinline__ Acc tile_prefix(const LookBack &lb, int64_t tile, int64_t first, Acc agg,
                                           Acc *sm_prefix) {
    publish_aggregate<Acc, Op>(lb, tile, first, agg);
    return lookback_prefix<Acc, Op>(lb, tile, first, agg, sm_prefix);
}

}  // namespace mt
