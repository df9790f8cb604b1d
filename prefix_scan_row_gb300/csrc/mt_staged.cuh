// mt_staged.cuh -- persistent scan over shared-memory-staged super-tiles.
//
// Each loop iteration of a CTA:
//   1. takes the next super-tile id (an atomic counter: a tile is only taken
//      when its load starts, so every tile waited on is already loading) and
//      issues one bulk copy (TMA) of the super-tile into shared memory;
//   2. computes the super-tile's aggregate with a quick reduction and
//      publishes it at once, so that later tiles' look-backs wait less;
//   3. scans it in SUB sub-tiles of THREADS x ITEMS 16-byte chunks (registers,
//      warp shuffles, block totals) with a running carry across sub-tiles, and
//      writes each element's super-tile-local prefix back to shared memory
//      in place;
//   4. looks back for the super-tile's prefix (one look-back per SUB
//      sub-tiles), combines it with the local prefixes and stores the outputs.
// The super-tile makes look-backs SUB times rarer per byte, and the input in
// flight per SM is (resident CTAs) x (super-tile bytes) without spending
// registers on it. Every super-tile but the first and last of a segment lies
// wholly inside it; those take a path with no per-chunk range checks.
// Types whose arithmetic, not memory, bounds the scan (f64: GB300 issues
// FP64 adds at about 2 per clock per SM) take a leaner form of steps 2-4,
// tile_lean: per-thread runs of consecutive chunks and about 2 combines per
// element instead of 5 to 7.
#pragma once

#include <type_traits>

#include "mt_lookback.cuh"

namespace mt {

// One scan call: nseg segments (rows) of n elements each, cut into tpr
// super-tiles per segment; or one 1-D array whose live count is n_dev.
struct SegArgs {
    const char *in;
    char *out;
    int64_t nseg;                 // number of segments (rows); 1 for a 1-D array
    int64_t n;                    // elements per segment (unused when n_dev is set)
    int64_t tpr;                  // super-tiles per segment (unused when n_dev is set)
    const int32_t *n_dev;         // 1-D: the live count, read on the device
    unsigned long long *counter;  // dynamic tile ids; nullptr: static assignment
    int inclusive;
    int aligned_io;               // output has the input's 16-byte phase
    LookBack lb;                  // lb.recs == nullptr: no tile waits on another
    const char *out_end;          // one past the call's output (set by the kernel; checked build)
};

#ifndef MT_STAGED_WAIT_WARP0
#define MT_STAGED_WAIT_WARP0 1  // only warp 0 polls the copy's mbarrier
#endif
#ifndef MT_STAGED_PAIR_W4
#define MT_STAGED_PAIR_W4 1  // scan 4-byte types two chunks per thread unit
#endif
#ifndef MT_STAGED_PAIR_W8
#define MT_STAGED_PAIR_W8 1  // the same for 8-byte types
#endif
#ifndef MT_STAGED_EARLY_W4
#define MT_STAGED_EARLY_W4 1  // early aggregate for 4-byte accumulators
#endif
#ifndef MT_STAGED_EARLY_W8
#define MT_STAGED_EARLY_W8 1  // the same for 8-byte accumulators
#endif
#ifndef MT_STAGED_LEAN_F64
#define MT_STAGED_LEAN_F64 1  // f64: per-thread runs (tile_lean)
#endif

template <class S, class Op, int ITEMS, int SUB, int THREADS>
struct Staged {
    using C = Codec<S>;
    using Acc = typename C::Acc;
    static constexpr int E = C::E;
    static constexpr int kNW = THREADS / 32;
    static constexpr int kSubChunks = THREADS * ITEMS;      // chunks per sub-tile
    static constexpr int kChunks = SUB * kSubChunks;        // chunks per super-tile
    static constexpr int64_t kTE = (int64_t)kChunks * E;    // virtual elements per super-tile
    // local prefixes of one chunk, in 16-byte planes: 1 when Acc is as wide as S
    static constexpr int kPlanes = (E * (int)sizeof(Acc) + 15) / 16;
    static constexpr int kPerPlane = 16 / (int)sizeof(Acc);  // Acc values per plane
    // Pass 1 scans units of V adjacent chunks per thread: a longer serial
    // run per thread and V times fewer warp scans per element. V = 2 needs
    // one plane (prefixes as wide as the input) and an even ITEMS.
    static constexpr int V =
        (kPlanes == 1 && ITEMS % 2 == 0 && (sizeof(Acc) == 8 ? MT_STAGED_PAIR_W8 : MT_STAGED_PAIR_W4)) ? 2 : 1;
    // Types whose combines, not memory, bound the scan take tile_lean: on
    // GB300 an f64 add issues at about 2 per clock per SM. (64-bit integers
    // were measured slower in that form: memory bounds them.)
    static constexpr bool kLean = kPlanes == 1 && std::is_same<Acc, double>::value && MT_STAGED_LEAN_F64;
    static constexpr int kRun = kChunks / THREADS;  // tile_lean: chunks per thread, consecutive
    static constexpr int kU = ITEMS / V;  // units per thread per sub-tile
    static constexpr int EU = V * E;      // elements per unit

    struct Smem {
        uint4 stage[kChunks];                                    // input; plane 0 of the prefixes
        uint4 extra[kPlanes > 1 ? (kPlanes - 1) * kChunks : 1];  // further planes
        uint64_t bar;
        int64_t tile;
        Acc warp_tot[2][kNW];
        Acc red[SUB][kNW];  // per-warp totals of the early reduction
        Acc prefix[2];
    };
    static constexpr size_t kSmemBytes = sizeof(Smem);

    // Chunk index of this thread's j-th chunk of sub-tile `sub`.
    __device__ __forceinline__ static int chunk_of(int sub, int j) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        return sub * kSubChunks + warp * 32 * ITEMS + j * 32 + lane;
    }

    // Chunk c of the staged input, widened. Without FULL, elements outside
    // the in-tile range [llo, lhi) become the identity (their stage bytes may
    // be stale: the copy only covers chunks that hold valid elements).
    template <bool FULL>
    __device__ __forceinline__ static void load(const Smem &sm, int c, int llo, int lhi, Acc (&x)[E]) {
        C::unpack(MT_CHECK_INDEX(c, kChunks) ? lds128(&sm.stage[c]) : make_uint4(0u, 0u, 0u, 0u), x);
        if (!FULL) {
            const int o = c * E;
            if (!(o >= llo && o + E <= lhi)) {
                const Acc ident = Op::template identity<Acc>();
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (o + k < llo || o + k >= lhi)
                        x[k] = ident;
            }
        }
    }

    __device__ __forceinline__ static uint4 *plane(Smem &sm, int p, int c) {
        return p == 0 ? &sm.stage[c] : &sm.extra[(p - 1) * kChunks + c];
    }
    __device__ __forceinline__ static void put(Smem &sm, int c, const Acc (&x)[E]) {
#pragma unroll
        for (int p = 0; p < kPlanes; ++p) {
            uint4 w;
            Acc *d = reinterpret_cast<Acc *>(&w);
#pragma unroll
            for (int r = 0; r < kPerPlane; ++r)
                d[r] = (p * kPerPlane + r < E) ? x[p * kPerPlane + r] : Acc(0);
            if (MT_CHECK_INDEX(c, kChunks))
                sts128(plane(sm, p, c), w);
        }
    }
    __device__ __forceinline__ static void get(Smem &sm, int c, Acc (&x)[E]) {
#pragma unroll
        for (int p = 0; p < kPlanes; ++p) {
            const uint4 w = MT_CHECK_INDEX(c, kChunks) ? lds128(plane(sm, p, c)) : make_uint4(0u, 0u, 0u, 0u);
            const Acc *d = reinterpret_cast<const Acc *>(&w);
#pragma unroll
            for (int r = 0; r < kPerPlane; ++r)
                if (p * kPerPlane + r < E)
                    x[p * kPerPlane + r] = d[r];
        }
    }

    // Unit index of this thread's j-th unit of sub-tile `sub`; its chunks
    // are V * unit ... V * unit + V - 1.
    __device__ __forceinline__ static int unit_of(int sub, int j) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        return sub * (kSubChunks / V) + warp * 32 * kU + j * 32 + lane;
    }
    // With V = 2, lanes 4-7 of every group of 8 take their unit's second
    // chunk first: the 8 lanes that share a shared-memory wavefront then
    // touch 8 different 16-byte bank groups, for loads and stores alike.
    __device__ __forceinline__ static int pair_swap() { return (threadIdx.x >> 2) & 1; }
    __device__ __forceinline__ static uint4 pick(bool s, const uint4 &a, const uint4 &b) {
        return make_uint4(s ? a.x : b.x, s ? a.y : b.y, s ? a.z : b.z, s ? a.w : b.w);
    }
    template <bool FULL>
    __device__ __forceinline__ static void load_unit(const Smem &sm, int u, int llo, int lhi, Acc (&x)[EU]) {
        if constexpr (V == 1) {
            load<FULL>(sm, u, llo, lhi, x);
        } else {
            const bool s = pair_swap();
            const bool in = MT_CHECK_INDEX(2 * u + 1, kChunks) && MT_CHECK_INDEX(2 * u, kChunks);
            const uint4 p = in ? lds128(&sm.stage[2 * u + (s ? 1 : 0)]) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 q = in ? lds128(&sm.stage[2 * u + (s ? 0 : 1)]) : make_uint4(0u, 0u, 0u, 0u);
            Acc lo[E], hi[E];
            C::unpack(pick(s, q, p), lo);
            C::unpack(pick(s, p, q), hi);
#pragma unroll
            for (int k = 0; k < E; ++k) {
                x[k] = lo[k];
                x[E + k] = hi[k];
            }
            if (!FULL) {
                const int o = u * EU;
                if (!(o >= llo && o + EU <= lhi)) {
                    const Acc ident = Op::template identity<Acc>();
#pragma unroll
                    for (int k = 0; k < EU; ++k)
                        if (o + k < llo || o + k >= lhi)
                            x[k] = ident;
                }
            }
        }
    }
    __device__ __forceinline__ static void put_unit(Smem &sm, int u, const Acc (&x)[EU]) {
        if constexpr (V == 1) {
            put(sm, u, x);
        } else {
            uint4 w[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                Acc *d = reinterpret_cast<Acc *>(&w[q]);
#pragma unroll
                for (int r = 0; r < E; ++r)
                    d[r] = x[q * E + r];
            }
            const bool s = pair_swap();
            if (MT_CHECK_INDEX(2 * u + 1, kChunks) && MT_CHECK_INDEX(2 * u, kChunks)) {
                sts128(&sm.stage[2 * u + (s ? 1 : 0)], pick(s, w[1], w[0]));
                sts128(&sm.stage[2 * u + (s ? 0 : 1)], pick(s, w[0], w[1]));
            }
        }
    }

    // The super-tile's aggregate (valid in every thread). Any grouping gives
    // the same result for adds of integers, for integer min/max, and for float
    // min/max unless the result is a zero (which of +0/-0 comes first then
    // matters): those take the quick unordered reduction, and a float min/max
    // whose quick result is zero is redone in element order. Float adds and
    // products take the quick one too (only rounding differs, within the
    // stated tolerances).
    template <bool FULL>
    __device__ __forceinline__ static Acc reduce(Smem &sm, int llo, int lhi) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();
        Acc acc = ident;
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                Acc x[E];
                load<FULL>(sm, chunk_of(sub, j), llo, lhi, x);
#pragma unroll
                for (int k = 0; k < E; ++k)
                    acc = Op::apply(acc, x[k]);
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            acc = Op::apply(acc, __shfl_xor_sync(kFull, acc, d));
        if (lane == 0)
            sm.red[0][warp] = acc;
        __syncthreads();
        Acc agg = ident;
#pragma unroll
        for (int w = 0; w < kNW; ++w)
            agg = Op::apply(agg, sm.red[0][w]);
        constexpr bool kOrderFree = std::is_same<Op, OpAdd>::value || std::is_same<Op, OpMul>::value ||
                                    !std::is_floating_point<Acc>::value;
        if constexpr (!kOrderFree) {
            if (agg == Acc(0)) {  // block-uniform: every thread folded the same totals
                __syncthreads();  // all reads of sm.red are done
#pragma unroll 1
                for (int sub = 0; sub < SUB; ++sub) {
                    Acc r = ident;
#pragma unroll
                    for (int j = 0; j < ITEMS; ++j) {
                        Acc x[E];
                        load<FULL>(sm, chunk_of(sub, j), llo, lhi, x);
                        Acc c = x[0];
#pragma unroll
                        for (int k = 1; k < E; ++k)
                            c = Op::apply(c, x[k]);
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {  // lane order: lower lanes are earlier
                            const Acc o = __shfl_down_sync(kFull, c, d);
                            if (lane + d < 32)
                                c = Op::apply(c, o);
                        }
                        r = Op::apply(r, c);
                    }
                    if (lane == 0)
                        sm.red[sub][warp] = r;
                }
                __syncthreads();
                agg = ident;
                for (int sub = 0; sub < SUB; ++sub)
                    for (int w = 0; w < kNW; ++w)
                        agg = Op::apply(agg, sm.red[sub][w]);
            }
        }
        return agg;
    }

    // One super-tile in per-thread runs, for accumulators whose combine is
    // the bound: thread t owns the kRun consecutive chunks from t * kRun.
    // Pass 0 folds the run serially; one warp scan of the run totals; warp 0
    // scans the warp totals, publishes the aggregate and looks back; pass 1
    // scans the run again from the thread's full prefix and writes the final
    // values in place; a last pass stores them chunk-coalesced. That is 2
    // combines per element plus about 7 per run (the sub-tile form takes
    // 5 to 7 per element). Every combine is in element order, so min and max
    // give the serial result bit for bit.
    template <bool FULL>
    __device__ __forceinline__ static void tile_lean(Smem &sm, const SegArgs &a, int64_t g, int64_t first,
                                                     S *eo, int llo, int lhi, int buf) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();
        const int cb = threadIdx.x * kRun;

        // Pass 0: the run's total.
        Acc tot;
        {
            Acc x[E];
            load<FULL>(sm, cb, llo, lhi, x);
            tot = x[0];
#pragma unroll
            for (int k = 1; k < E; ++k)
                tot = Op::apply(tot, x[k]);
        }
#pragma unroll
        for (int j = 1; j < kRun; ++j) {
            Acc x[E];
            load<FULL>(sm, cb + j, llo, lhi, x);
#pragma unroll
            for (int k = 0; k < E; ++k)
                tot = Op::apply(tot, x[k]);
        }

        // The runs' exclusive prefixes within the warp.
        Acc inc = tot;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const Acc y = __shfl_up_sync(kFull, inc, d);
            if (lane >= d)
                inc = Op::apply(y, inc);
        }
        Acc ex = __shfl_up_sync(kFull, inc, 1);
        if (lane == 0)
            ex = ident;
        if (lane == 31)
            sm.warp_tot[0][warp] = inc;
        __syncthreads();

        // Warp 0: the warps' exclusive prefixes, the aggregate (published
        // at once), the look-back, the inclusive prefix.
        if (warp == 0) {
            Acc w = lane < kNW ? sm.warp_tot[0][lane] : ident;
#pragma unroll
            for (int d = 1; d < kNW; d <<= 1) {
                const Acc y = __shfl_up_sync(kFull, w, d);
                if (lane >= d)
                    w = Op::apply(y, w);
            }
            Acc wex = __shfl_up_sync(kFull, w, 1);
            if (lane == 0)
                wex = ident;
            const Acc agg = __shfl_sync(kFull, w, kNW - 1);
            if (lane < kNW)
                sm.warp_tot[1][lane] = wex;
            publish_aggregate<Acc, Op>(a.lb, g, first, agg);
            Acc pre = ident;
            if (a.lb.recs != nullptr && g != first) {
                pre = warp_lookback<Acc, Op>(a.lb.recs, g, first, a.lb.spin_limit);
                if (lane == 0 && g != a.lb.skip_tile)
                    publish_record<Acc>(a.lb, g, kIncl, Op::apply(pre, agg));
            }
            if (lane == 0)
                sm.prefix[buf] = pre;
        }
        __syncthreads();

        // Pass 1: the run scanned from its full prefix, in place.
        Acc run = Op::apply(Op::apply(sm.prefix[buf], sm.warp_tot[1][warp]), ex);
#pragma unroll
        for (int j = 0; j < kRun; ++j) {
            Acc x[E];
            load<FULL>(sm, cb + j, llo, lhi, x);
            if (a.inclusive) {
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    run = Op::apply(run, x[k]);
                    x[k] = run;
                }
            } else {
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const Acc v = x[k];
                    x[k] = run;
                    run = Op::apply(run, v);
                }
            }
            put(sm, cb + j, x);
        }
        __syncthreads();

        // Stores: consecutive lanes on consecutive chunks.
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const int c = chunk_of(sub, j);
                const int o = c * E;
                if (!FULL && !(o < lhi && o + E > llo))
                    continue;
                const uint4 w = MT_CHECK_INDEX(c, kChunks) ? lds128(&sm.stage[c]) : make_uint4(0u, 0u, 0u, 0u);
                if (a.aligned_io && (FULL || (o >= llo && o + E <= lhi))) {
                    uint4 *p = reinterpret_cast<uint4 *>(eo) + c;
                    if (MT_CHECK_RANGE(p, 16, a.out, a.out_end))
                        st_v4(p, w);
                } else {
                    Acc x[E];
                    C::unpack(w, x);
#pragma unroll
                    for (int k = 0; k < E; ++k)
                        if ((FULL || (o + k >= llo && o + k < lhi)) && MT_CHECK_RANGE(eo + o + k, sizeof(S), a.out, a.out_end))
                            C::store1(eo + o + k, x[k]);
                }
            }
        }
    }

    // One super-tile, from the staged input to the stored outputs.
    //   eo        : output address of the super-tile's virtual element 0
    //   [llo, lhi): the super-tile's valid elements ([0, kTE) when FULL)
    //   g / first : the super-tile's id and the id of its segment's first one
    //   buf       : which half of the double-buffered prefix slot to use
    template <bool FULL>
    __device__ __forceinline__ static void tile(Smem &sm, const SegArgs &a, int64_t g, int64_t first,
                                                S *eo, int llo, int lhi, int buf) {
        if constexpr (kLean) {
            tile_lean<FULL>(sm, a, g, first, eo, llo, lhi, buf);
            return;
        }
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();

        // Pass 0: the aggregate, published before the scan.
        constexpr bool kEarly = sizeof(Acc) == 8 ? MT_STAGED_EARLY_W8 : MT_STAGED_EARLY_W4;
        Acc agg_total = ident;
        if constexpr (kEarly) {
            agg_total = reduce<FULL>(sm, llo, lhi);
            publish_aggregate<Acc, Op>(a.lb, g, first, agg_total);
        }

        // Pass 1: sub-tiles in order with a running carry; keep each
        // element's super-tile-local prefix in shared memory. (Looking back
        // first and storing final values from here saves pass 2's combine per
        // element but exposes the look-back's latency: measured slower
        // wherever memory bounds the kernel.)
        Acc carry = ident;
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
            Acc x[kU][EU];
#pragma unroll
            for (int j = 0; j < kU; ++j)
                load_unit<FULL>(sm, unit_of(sub, j), llo, lhi, x[j]);
            Acc inc[kU];
#pragma unroll
            for (int j = 0; j < kU; ++j) {
#pragma unroll
                for (int k = 1; k < EU; ++k)
                    x[j][k] = Op::apply(x[j][k - 1], x[j][k]);
                inc[j] = x[j][EU - 1];
            }
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
                for (int j = 0; j < kU; ++j) {
                    const Acc y = __shfl_up_sync(kFull, inc[j], d);
                    if (lane >= d)
                        inc[j] = Op::apply(y, inc[j]);
                }
            }
            Acc pre[kU];
            Acc run = ident;
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                Acc e = __shfl_up_sync(kFull, inc[j], 1);
                if (lane == 0)
                    e = ident;
                pre[j] = Op::apply(run, e);
                run = Op::apply(run, __shfl_sync(kFull, inc[j], 31));
            }
            if (lane == 0)
                sm.warp_tot[sub & 1][warp] = run;
            __syncthreads();
            // The warp totals scanned across the first kNW lanes (3 steps
            // instead of 2 kNW combines per thread), in warp order.
            Acc t = lane < kNW ? sm.warp_tot[sub & 1][lane] : ident;
#pragma unroll
            for (int d = 1; d < kNW; d <<= 1) {
                const Acc y = __shfl_up_sync(kFull, t, d);
                if (lane >= d)
                    t = Op::apply(y, t);
            }
            Acc wpre = __shfl_sync(kFull, t, (warp + 31) & 31);
            if (warp == 0)
                wpre = ident;
            const Acc agg = __shfl_sync(kFull, t, kNW - 1);
            const Acc base0 = Op::apply(carry, wpre);
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                const Acc base = Op::apply(base0, pre[j]);
                if (a.inclusive) {
#pragma unroll
                    for (int k = 0; k < EU; ++k)
                        x[j][k] = Op::apply(base, x[j][k]);
                } else {
#pragma unroll
                    for (int k = EU - 1; k > 0; --k)
                        x[j][k] = Op::apply(base, x[j][k - 1]);
                    x[j][0] = base;
                }
                put_unit(sm, unit_of(sub, j), x[j]);
            }
            carry = Op::apply(carry, agg);
        }

        if constexpr (!kEarly) {
            agg_total = carry;
            publish_aggregate<Acc, Op>(a.lb, g, first, agg_total);
        }

        // The super-tile's prefix: look back, publish the inclusive prefix
        // (the identity for a segment's first super-tile).
        const Acc tp = lookback_prefix<Acc, Op>(a.lb, g, first, agg_total, &sm.prefix[buf]);
        // Pass 2 reads chunks that other threads' units wrote when V > 1; the
        // look-back ends with a block barrier except for a segment's first
        // super-tile (or when no tile waits on another).
        if (V > 1 && (a.lb.recs == nullptr || g == first))
            __syncthreads();

        // Pass 2: prefix + local prefix, narrowed to S and stored; 16-byte
        // stores for whole chunks when the output has the input's phase.
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const int c = chunk_of(sub, j);
                const int o = c * E;
                if (!FULL && !(o < lhi && o + E > llo))
                    continue;
                Acc x[E];
                get(sm, c, x);
#pragma unroll
                for (int k = 0; k < E; ++k)
                    x[k] = Op::apply(tp, x[k]);
                if (a.aligned_io && (FULL || (o >= llo && o + E <= lhi))) {
                    uint4 *p = reinterpret_cast<uint4 *>(eo) + c;
                    if (MT_CHECK_RANGE(p, 16, a.out, a.out_end))
                        st_v4(p, C::pack(x));
                } else {
#pragma unroll
                    for (int k = 0; k < E; ++k)
                        if ((FULL || (o + k >= llo && o + k < lhi)) && MT_CHECK_RANGE(eo + o + k, sizeof(S), a.out, a.out_end))
                            C::store1(eo + o + k, x[k]);
                }
            }
        }
    }
};

template <class S, class Op, int ITEMS, int SUB, int THREADS>
__global__ void __launch_bounds__(THREADS, 65536 / (THREADS * 64)) k_scan_staged(SegArgs a) {
    pdl_prologue();
    using G = Staged<S, Op, ITEMS, SUB, THREADS>;
    constexpr int E = G::E;
    extern __shared__ __align__(128) unsigned char dsm[];
    typename G::Smem &sm = *reinterpret_cast<typename G::Smem *>(dsm);
    constexpr int64_t s = sizeof(S);

    int64_t n, tpr, ntiles;
    if (a.n_dev != nullptr) {
        const int32_t n32 = *a.n_dev;
        n = n32 > 0 ? n32 : 0;
        const int64_t head = (int64_t)(((uintptr_t)a.in & 15u) / s);
        tpr = n > 0 ? (head + n + G::kTE - 1) / G::kTE : 1;
        ntiles = n > 0 ? tpr : 0;
    } else {
        n = a.n;
        tpr = a.tpr;
        ntiles = a.nseg * tpr;
    }
    a.lb.nrec = ntiles;
    a.out_end = a.out + (a.n_dev != nullptr ? n : a.nseg * n) * s;

    if (threadIdx.x == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    uint32_t phase = 0;
    for (int64_t it = 0;; ++it) {
        if (threadIdx.x == 0)
            sm.tile = a.counter != nullptr ? (int64_t)atomicAdd(a.counter, 1ull)
                                           : (int64_t)blockIdx.x + it * (int64_t)gridDim.x;
        __syncthreads();  // tile id visible; every thread is done with the last super-tile
        const int64_t g = sm.tile;
        if (g >= ntiles)
            break;
        // Geometry of the super-tile inside its segment.
        const int64_t row = g / tpr;
        const int64_t kk = g - row * tpr;
        const char *in_row = a.in + row * n * s;
        const int64_t head = (int64_t)(((uintptr_t)in_row & 15u) / s);
        const uint4 *vin = reinterpret_cast<const uint4 *>(in_row - head * s);
        S *eout = reinterpret_cast<S *>(a.out + row * n * s) - head;
        const int64_t t0 = kk * G::kTE, lo = head, hi = head + n, first = row * tpr;
        const int64_t c0 = t0 / E;
        int64_t cend = (hi + E - 1) / E;
        if (cend > c0 + G::kChunks)
            cend = c0 + G::kChunks;
        if (cend <= c0) {  // a trailing super-tile past the row's end: nobody waits on it
            __syncthreads();  // every thread has read sm.tile before it is rewritten
            continue;
        }

        if (threadIdx.x == 0) {
            fence_proxy_async_smem();  // the last iteration's shared-memory writes come first
            uint32_t bytes = (uint32_t)((cend - c0) * 16);
            if (!MT_CHECK_RANGE(&sm.stage[0], bytes, &sm.stage[0], &sm.stage[G::kChunks]))
                bytes = 0u;  // checked build: no copy (the phase completes with no bytes)
            mbar_arrive_expect_tx(&sm.bar, bytes);
            if (bytes != 0u)
                bulk_g2s(&sm.stage[0], vin + c0, bytes, &sm.bar);
        }
        // Warp 0 waits for the copy; the block barrier then passes the
        // completion (and the copied bytes) on to the other warps.
        bool ok = true;
        if (!MT_STAGED_WAIT_WARP0 || threadIdx.x < 32)
            ok = mbar_wait(&sm.bar, phase, kCopyWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) {
                atomicCAS(&g_mt_err, 0, kErrTimeout);
                mbar_wait(&sm.bar, phase, kCopyWaitLimit);  // drain the copy before leaving
            }
            return;
        }
        phase ^= 1u;

        S *eo = eout + t0;
        const int buf = (int)(it & 1);
        if (t0 >= lo && t0 + G::kTE <= hi) {
            G::template tile<true>(sm, a, g, first, eo, 0, (int)G::kTE, buf);
        } else {
            const int llo = lo > t0 ? (int)(lo - t0) : 0;
            const int lhi = hi - t0 < G::kTE ? (int)(hi - t0) : (int)G::kTE;
            G::template tile<false>(sm, a, g, first, eo, llo, lhi, buf);
        }
        fence_proxy_async_smem();  // this thread's shared writes precede the next bulk copy
    }
}

template <class S, class Op, int ITEMS, int SUB, int THREADS>
static cudaError_t launch_staged(const SegArgs &a, int64_t max_ctas, const Launch &L) {
    using G = Staged<S, Op, ITEMS, SUB, THREADS>;
    static PerDevice per_sm;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int blocks = per_sm.get(dev);
    if (blocks == 0) {
        e = cudaFuncSetAttribute(k_scan_staged<S, Op, ITEMS, SUB, THREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        // the whole unified L1/shared array as shared memory, so that as many
        // super-tiles as registers allow are in flight on each SM
        e = cudaFuncSetAttribute(k_scan_staged<S, Op, ITEMS, SUB, THREADS>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_scan_staged<S, Op, ITEMS, SUB, THREADS>,
                                                          THREADS, G::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        blocks = b > 0 ? b : 1;
        per_sm.set(dev, blocks);
    }
    int64_t grid = (int64_t)L.sm_count * blocks;
    if (max_ctas > 0 && grid > max_ctas)
        grid = max_ctas;
    if (grid < 1)
        grid = 1;
    e = launch_pdl(k_scan_staged<S, Op, ITEMS, SUB, THREADS>, (unsigned)grid, THREADS, G::kSmemBytes,
                   L.stream, a);
    note_launch();
    return e;
}

}  // namespace mt
