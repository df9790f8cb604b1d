// mt_tilescan.cuh -- one CTA tile of a scan over storage type S with combine Op.
//
// Addressing uses "virtual elements": element 0 of a segment sits at virtual
// index `head` = (start address mod 16) / sizeof(S) counted from the 16-byte
// boundary below it. Chunk c covers virtual [c*E, c*E + E), so every vector
// access is 16-byte aligned whatever the row start. Virtual elements outside
// the segment's valid range [lo, hi) are loaded (the aligned 16-byte chunk
// around a valid element lies in the same page) but enter the scan as the
// identity and are never stored.
#pragma once

#include "mt_lookback.cuh"

namespace mt {

template <class S, class Op, int ITEMS>
struct TileScan {
    using C = Codec<S>;
    using Acc = typename C::Acc;
    static constexpr int E = C::E;
    static constexpr int kChunks = kThreads * ITEMS;
    static constexpr int64_t kTE = (int64_t)kChunks * E;  // virtual elements per tile

    struct Smem {
        Acc warp_tot[kWarps];
        Acc prefix;
        unsigned long long tile;
    };

    __device__ __forceinline__ static int64_t chunk_v(int64_t t0, int j) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        return t0 + (int64_t)(warp * 32 * ITEMS + j * 32 + lane) * E;
    }

    // Scan the tile covering virtual [t0, t0 + kTE) of a segment.
    //   vin       : 16-byte aligned address of virtual element 0 of the input
    //   eout      : address of virtual element 0 of the output (element pointer)
    //   aligned_io: eout is 16-byte aligned too (same phase as the input)
    //   [lo, hi)  : valid virtual range of the segment
    //   tile/first: global tile id and the id of the segment's first tile
    __device__ __forceinline__ static void run(const uint4 *vin, S *eout, bool aligned_io, int64_t t0,
                                               int64_t lo, int64_t hi, bool inclusive,
                                               const LookBack &lb, int64_t tile, int64_t first,
                                               Smem &sm) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();

        // 1. Issue every load of the tile before using any of them.
        uint4 raw[ITEMS];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int64_t v = chunk_v(t0, j);
            raw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (v < hi && v + E > lo)
                raw[j] = ld_stream(vin + v / E);
        }
        Acc x[ITEMS][E];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int64_t v = chunk_v(t0, j);
            C::unpack(raw[j], x[j]);
            if (!(v >= lo && v + E <= hi)) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (v + k < lo || v + k >= hi)
                        x[j][k] = ident;
            }
        }

        // 2. Inclusive scan of each chunk in registers.
        Acc inc[ITEMS];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
#pragma unroll
            for (int k = 1; k < E; ++k)
                x[j][k] = Op::apply(x[j][k - 1], x[j][k]);
            inc[j] = x[j][E - 1];
        }

        // 3. Inclusive warp scans of the chunk totals (one per j, interleaved).
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const Acc y = __shfl_up_sync(kFull, inc[j], d);
                if (lane >= d)
                    inc[j] = Op::apply(y, inc[j]);
            }
        }

        // 4. Prefix of each chunk inside the warp's run; the warp total.
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
            sm.warp_tot[warp] = run;
        __syncthreads();

        // 5. Block: this warp's exclusive prefix and the tile aggregate.
        Acc wpre = ident, agg = ident;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const Acc t = sm.warp_tot[w];
            if (w < warp)
                wpre = Op::apply(wpre, t);
            agg = Op::apply(agg, t);
        }

        // 6. Tile prefix from the look-back (identity for a segment's first tile).
        const Acc tp = tile_prefix<Acc, Op>(lb, tile, first, agg, &sm.prefix);
        const Acc base0 = Op::apply(tp, wpre);

        // 7. Outputs: inclusive base + s_k, or exclusive base + s_{k-1} with
        //    base itself at k = 0 (the one-slot shift of scan.rs's exclusive
        //    kernel).
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
            const int64_t v = chunk_v(t0, j);
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
};

}  // namespace mt
