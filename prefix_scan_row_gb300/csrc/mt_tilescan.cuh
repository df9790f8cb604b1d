// mt_tilescan.cuh -- one row scanned by one CTA in a single tile.
//
// Addressing uses "virtual elements": element 0 of a row sits at virtual
// index `head` = (start address mod 16) / sizeof(S) counted from the 16-byte
// boundary below it. Chunk c covers virtual [c*E, c*E + E), so every vector
// access is 16-byte aligned whatever the row start. Virtual elements outside
// the row's valid range [lo, hi) are loaded (the aligned 16-byte chunk around
// a valid element lies in the same page) but enter the scan as the identity
// and are never stored. A row that fills its tile exactly (lo == 0 and
// hi == the tile's size) takes a path with no range checks at all.
//
// The block size is taken from blockDim at run time (at most 16 warps), so
// one instantiation per chunks-per-thread count serves every row length.
#pragma once

#include "mt_lookback.cuh"

namespace mt {

template <class S, class Op, int ITEMS>
struct RowTile {
    using C = Codec<S>;
    using Acc = typename C::Acc;
    static constexpr int E = C::E;
    static constexpr int kMaxWarps = 16;

    struct Smem {
        Acc warp_tot[kMaxWarps];
    };

    // Index of chunk j of this thread inside the tile.
    __device__ __forceinline__ static int chunk_of(int j) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        return warp * 32 * ITEMS + j * 32 + lane;
    }

    // Scan the tile (virtual [0, 32 * warps * ITEMS * E)) and store it.
    //   vin       : the row's input from its 16-byte boundary (chunk pointer)
    //   eout      : output address of virtual element 0 (element pointer)
    //   aligned_io: eout is 16-byte aligned (same phase as the input)
    //   [lo, hi)  : the row's valid virtual range; FULL: all of the tile
    //   [olo, ohi): the row's output bytes (every store is checked against
    //               them in a bounds-checked build)
    template <bool FULL>
    __device__ __forceinline__ static void run(const uint4 *vin, S *eout, bool aligned_io, int lo, int hi,
                                               bool inclusive, Smem &sm, const char *olo, const char *ohi) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();

        // Every load is issued before any is used.
        uint4 raw[ITEMS];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int o = chunk_of(j) * E;
            if (FULL) {
                raw[j] = ld_stream(vin + chunk_of(j));
            } else {
                raw[j] = make_uint4(0u, 0u, 0u, 0u);
                if (o < hi && o + E > lo)
                    raw[j] = ld_stream(vin + chunk_of(j));
            }
        }

        Acc x[ITEMS][E];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            C::unpack(raw[j], x[j]);
            if (!FULL) {
                const int o = chunk_of(j) * E;
                if (!(o >= lo && o + E <= hi)) {
#pragma unroll
                    for (int k = 0; k < E; ++k)
                        if (o + k < lo || o + k >= hi)
                            x[j][k] = ident;
                }
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
        if (lane == 0 && MT_CHECK_INDEX(warp, kMaxWarps))
            sm.warp_tot[warp] = run;
        __syncthreads();

        // This warp's exclusive prefix: the totals of the warps before it.
        const int nw = (int)(blockDim.x >> 5);
        Acc t = lane < nw ? sm.warp_tot[lane] : ident;
#pragma unroll
        for (int d = 1; d < kMaxWarps; d <<= 1) {
            const Acc y = __shfl_up_sync(kFull, t, d);
            if (lane >= d)
                t = Op::apply(y, t);
        }
        Acc wpre = __shfl_sync(kFull, t, (warp + 31) & 31);
        if (warp == 0)
            wpre = ident;

        // Outputs: inclusive base + s_k, or exclusive base + s_{k-1} with base
        // itself at k = 0 (the one-slot shift of scan.rs's exclusive kernel).
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const Acc base = Op::apply(wpre, pre[j]);
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
            const int c = chunk_of(j);
            const int o = c * E;
            if (aligned_io && (FULL || (o >= lo && o + E <= hi))) {
                uint4 *p = reinterpret_cast<uint4 *>(eout) + c;
                if (MT_CHECK_RANGE(p, 16, olo, ohi))
                    st_v4(p, C::pack(x[j]));
            } else if (FULL || (o < hi && o + E > lo)) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if ((FULL || (o + k >= lo && o + k < hi)) && MT_CHECK_RANGE(eout + o + k, sizeof(S), olo, ohi))
                        C::store1(eout + o + k, x[j][k]);
            }
        }
    }
};

}  // namespace mt
