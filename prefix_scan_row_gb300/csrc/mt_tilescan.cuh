// mt_tilescan.cuh -- one CTA tile of a scan over storage type S with combine Op.
//
// Addressing uses "virtual elements": element 0 of a segment sits at virtual
// index `head` = (start address mod 16) / sizeof(S) counted from the 16-byte
// boundary below it. Chunk c covers virtual [c*E, c*E + E), so every vector
// access is 16-byte aligned whatever the row start. Virtual elements outside
// the segment's valid range [lo, hi) are loaded (the aligned 16-byte chunk
// around a valid element lies in the same page) but enter the scan as the
// identity and are never stored.
//
// A tile is scanned in two phases: a load phase (from global memory, or from
// a shared-memory stage filled by a bulk copy) into `raw` registers, and
// scan_store(), which scans, obtains the tile prefix and stores the outputs.
#pragma once

#include "mt_lookback.cuh"

namespace mt {

struct NoHook {
    __device__ __forceinline__ void operator()() const {}
};

// THREADS == 0: the block size is taken from blockDim at run time (at most
// 16 warps); kChunks and kTE are then not meaningful.
template <class S, class Op, int ITEMS, int THREADS = kThreads>
struct TileScan {
    using C = Codec<S>;
    using Acc = typename C::Acc;
    static constexpr int E = C::E;
    static constexpr bool kDyn = THREADS == 0;
    static constexpr int kNW = kDyn ? 16 : THREADS / 32;    // warps per CTA (the maximum when dynamic)
    static constexpr int kChunks = THREADS * ITEMS;
    static constexpr int64_t kTE = (int64_t)kChunks * E;  // virtual elements per tile
    static_assert(THREADS % 32 == 0 && THREADS <= 1024, "block size");

    struct Smem {
        Acc warp_tot[2][kNW];  // double-buffered: consecutive tiles of a persistent CTA
        Acc warp_pre[2][kNW];  // exclusive warp prefixes (more than 8 warps)
        Acc agg[2];
        Acc prefix[2];
        unsigned long long tile;
    };

    // Index of chunk j of this thread inside the tile.
    __device__ __forceinline__ static int chunk_of(int j) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        return warp * 32 * ITEMS + j * 32 + lane;
    }

    // Loads straight from global memory; every load is issued before any is used.
    __device__ __forceinline__ static void load_global(const uint4 *vin, int64_t t0, int64_t lo,
                                                       int64_t hi, uint4 (&raw)[ITEMS]) {
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int64_t v = t0 + (int64_t)chunk_of(j) * E;
            raw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (v < hi && v + E > lo)
                raw[j] = ld_stream(vin + v / E);
        }
    }

    // Loads from a shared-memory stage holding the tile's chunks in order
    // (chunk c at stage[c]); conflict-free (consecutive lanes, consecutive 16 B).
    __device__ __forceinline__ static void load_stage(const uint4 *stage, int64_t t0, int64_t lo,
                                                      int64_t hi, uint4 (&raw)[ITEMS]) {
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int c = chunk_of(j);
            const int64_t v = t0 + (int64_t)c * E;
            raw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (v < hi && v + E > lo)
                raw[j] = stage[c];
        }
    }

    // Scan the tile covering virtual [t0, t0 + kTE) of a segment and store it.
    //   eout      : address of virtual element 0 of the output (element pointer)
    //   aligned_io: eout is 16-byte aligned (same phase as the input)
    //   [lo, hi)  : valid virtual range of the segment
    //   tile/first: global tile id and the id of the segment's first tile
    //   buf       : which half of the double-buffered shared state to use
    //   hook      : run by every thread right after the block barrier that
    //               follows the last read of `raw`'s source (a stage may be
    //               refilled from there on)
    template <class Hook>
    __device__ __forceinline__ static void scan_store(uint4 (&raw)[ITEMS], S *eout, bool aligned_io,
                                                      int64_t t0, int64_t lo, int64_t hi,
                                                      bool inclusive, const LookBack &lb,
                                                      int64_t tile, int64_t first, Smem &sm, int buf,
                                                      const Hook &hook) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();

        Acc x[ITEMS][E];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int64_t v = t0 + (int64_t)chunk_of(j) * E;
            C::unpack(raw[j], x[j]);
            if (!(v >= lo && v + E <= hi)) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (v + k < lo || v + k >= hi)
                        x[j][k] = ident;
            }
        }

        // Inclusive scan of each chunk in registers.
        Acc inc[ITEMS];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
#pragma unroll
            for (int k = 1; k < E; ++k)
                x[j][k] = Op::apply(x[j][k - 1], x[j][k]);
            inc[j] = x[j][E - 1];
        }

        // Inclusive warp scans of the chunk totals (one per j, interleaved).
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const Acc y = __shfl_up_sync(kFull, inc[j], d);
                if (lane >= d)
                    inc[j] = Op::apply(y, inc[j]);
            }
        }

        // Prefix of each chunk inside the warp's run; the warp total.
        Acc pre[ITEMS];
        Acc run = ident;
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            Acc e = __shfl_up_sync(kFull, inc[j], 1);
            if (lane == 0)
                e = ident;
            pre[j] = Op::apply(run, e);
            run = Op::apply(run, __shfl_sync(kFull, inc[j], 31));
        }
        if (lane == 0)
            sm.warp_tot[buf][warp] = run;
        __syncthreads();
        hook();

        // Block: this warp's exclusive prefix and the tile aggregate.
        Acc wpre = ident, agg = ident;
        if constexpr (kDyn) {
            const int nw = blockDim.x >> 5;
            for (int w = 0; w < nw; ++w) {
                const Acc t = sm.warp_tot[buf][w];
                if (w < warp)
                    wpre = Op::apply(wpre, t);
                agg = Op::apply(agg, t);
            }
        } else if constexpr (kNW <= 8) {
            // few warps: every thread folds the warp totals itself
#pragma unroll
            for (int w = 0; w < kNW; ++w) {
                const Acc t = sm.warp_tot[buf][w];
                if (w < warp)
                    wpre = Op::apply(wpre, t);
                agg = Op::apply(agg, t);
            }
        } else {
            // many warps: warp 0 scans the totals, one more barrier
            if (warp == 0) {
                Acc t = lane < kNW ? sm.warp_tot[buf][lane] : ident;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const Acc y = __shfl_up_sync(kFull, t, d);
                    if (lane >= d)
                        t = Op::apply(y, t);
                }
                Acc e = __shfl_up_sync(kFull, t, 1);
                if (lane == 0)
                    e = ident;
                if (lane < kNW)
                    sm.warp_pre[buf][lane] = e;
                if (lane == 31)
                    sm.agg[buf] = t;
            }
            __syncthreads();
            wpre = sm.warp_pre[buf][warp];
            agg = sm.agg[buf];
        }

        // Tile prefix from the look-back (identity for a segment's first tile).
        const Acc tp = tile_prefix<Acc, Op>(lb, tile, first, agg, &sm.prefix[buf]);
        const Acc base0 = Op::apply(tp, wpre);

        // Outputs: inclusive base + s_k, or exclusive base + s_{k-1} with base
        // itself at k = 0 (the one-slot shift of scan.rs's exclusive kernel).
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const Acc base = Op::apply(base0, pre[j]);
            if (inclusive) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    x[j][k] = Op::apply(base, x[j][k]);
            } else {
#pragma unroll
                for (int k = E - 1; k > 0; --k)
                    x[j][k] = Op::apply(base, x[j][k - 1]);
                x[j][0] = base;
            }
            const int64_t v = t0 + (int64_t)chunk_of(j) * E;
            if (aligned_io && v >= lo && v + E <= hi) {
                st_v4(reinterpret_cast<uint4 *>(eout) + v / E, C::pack(x[j]));
            } else if (v < hi && v + E > lo) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (v + k >= lo && v + k < hi)
                        C::store1(eout + v + k, x[j][k]);
            }
        }
    }

    // One tile read straight from global memory (single-tile rows).
    __device__ __forceinline__ static void run(const uint4 *vin, S *eout, bool aligned_io, int64_t t0,
                                               int64_t lo, int64_t hi, bool inclusive,
                                               const LookBack &lb, int64_t tile, int64_t first,
                                               Smem &sm) {
        uint4 raw[ITEMS];
        load_global(vin, t0, lo, hi, raw);
        scan_store(raw, eout, aligned_io, t0, lo, hi, inclusive, lb, tile, first, sm, 0, NoHook());
    }
};

}  // namespace mt
