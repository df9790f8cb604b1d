// mt_staged.cuh -- persistent scan over shared-memory-staged super-tiles.
//
// Each loop iteration of a CTA:
//   1. takes the next super-tile id (an atomic counter: a tile is only taken
//      when its load starts, so every tile waited on is already loading) and
//      issues one bulk copy (TMA) of the super-tile into shared memory;
//   2. scans it in SUB sub-tiles of THREADS x ITEMS 16-byte chunks (registers,
//      warp shuffles, block totals) with a running carry across sub-tiles, and
//      writes each element's super-tile-local prefix back to shared memory --
//      every thread rereads only the chunks it wrote, so this needs no barrier;
//   3. publishes the super-tile aggregate -- computed by a quick reduction
//      before the scan, so other tiles' look-backs wait less -- and, after
//      the scan, looks back for its prefix (one look-back per SUB sub-tiles);
//   4. combines that prefix with the local prefixes and stores the outputs.
// The super-tile makes look-backs SUB times rarer per byte, and the input in
// flight per SM is (resident CTAs) x (super-tile bytes) without spending
// registers on it.
#pragma once

#include <type_traits>

#include "mt_tilescan.cuh"
#include "mt_pipe.cuh"

namespace mt {

#ifndef MT_STAGED_EARLY_LOOKBACK
#define MT_STAGED_EARLY_LOOKBACK 0  // 1: look back before the scan (one scan+store pass)
#endif

// A thread's group = V adjacent 16-byte chunks (V * E contiguous elements),
// scanned serially before the warp scan; V > 1 cuts the warp-scan work per
// element for wide element types.
template <class S, class Op, int ITEMS, int SUB, int THREADS, int V = 1>
struct Staged {
    using C = Codec<S>;
    using Acc = typename C::Acc;
    static constexpr int E = C::E;
    static constexpr int EG = E * V;                            // elements per group
    static constexpr int kNW = THREADS / 32;
    static constexpr int kSubGroups = THREADS * ITEMS;          // groups per sub-tile
    static constexpr int kSubChunks = kSubGroups * V;           // chunks per sub-tile
    static constexpr int kChunks = SUB * kSubChunks;            // chunks per super-tile
    static constexpr int64_t kTE = (int64_t)kChunks * E;        // virtual elements per super-tile
    // local prefixes of one chunk, in 16-byte planes: 1 when Acc is as wide as S
    static constexpr int kPlanes = MT_STAGED_EARLY_LOOKBACK ? 1 : (E * (int)sizeof(Acc) + 15) / 16;
    static constexpr int kPerPlane = 16 / (int)sizeof(Acc);     // Acc values per plane

    struct Smem {
        uint4 stage[kChunks];                          // input; plane 0 of the prefixes
        uint4 extra[kPlanes > 1 ? (kPlanes - 1) * kChunks : 1];  // further planes
        uint64_t bar;
        int64_t tile;
        Acc warp_tot[2][kNW];
        Acc red[SUB][kNW];  // per-warp totals of the early reduction
        Acc prefix[2];
    };
    static constexpr size_t kSmemBytes = sizeof(Smem);

    // Group index of this thread's j-th group of sub-tile `sub`; its chunks
    // are group * V ... group * V + V - 1.
    __device__ __forceinline__ static int chunk_of(int sub, int j) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        return sub * kSubGroups + warp * 32 * ITEMS + j * 32 + lane;
    }
    // Group gi of the staged input, widened, with elements outside [lo, hi)
    // replaced by the identity.
    __device__ __forceinline__ static void load_chunk(const Smem &sm, int gi, int64_t t0, int64_t lo,
                                                      int64_t hi, Acc (&x)[EG]) {
        const Acc ident = Op::template identity<Acc>();
        const int64_t v = t0 + (int64_t)gi * EG;
#pragma unroll
        for (int q = 0; q < V; ++q) {
            const int64_t vq = v + q * E;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (vq < hi && vq + E > lo)
                raw = sm.stage[gi * V + q];
            Acc part[E];
            C::unpack(raw, part);
#pragma unroll
            for (int k = 0; k < E; ++k)
                x[q * E + k] = part[k];
        }
        if (!(v >= lo && v + EG <= hi)) {
#pragma unroll
            for (int k = 0; k < EG; ++k)
                if (v + k < lo || v + k >= hi)
                    x[k] = ident;
        }
    }

    // The super-tile's aggregate (valid in thread 0). Any grouping gives the
    // same result for adds of integers, for integer min/max, and for float
    // min/max unless the result is a zero (which of +0/-0 comes first then
    // matters): those take the quick unordered reduction, and a float min/max
    // whose quick result is zero is redone in element order. Float adds take
    // the quick one too (only rounding differs, within the stated tolerance).
    __device__ __forceinline__ static Acc reduce(Smem &sm, int64_t t0, int64_t lo, int64_t hi) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const Acc ident = Op::template identity<Acc>();
        Acc acc = ident;
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                Acc x[EG];
                load_chunk(sm, chunk_of(sub, j), t0, lo, hi, x);
#pragma unroll
                for (int k = 0; k < EG; ++k)
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
        constexpr bool kOrderFree = std::is_same<Op, OpAdd>::value || !std::is_same<Acc, float>::value;
        if constexpr (!kOrderFree) {
            if (agg == Acc(0)) {  // block-uniform: every thread folded the same totals
                __syncthreads();  // all reads of sm.red are done
#pragma unroll 1
                for (int sub = 0; sub < SUB; ++sub) {
                    Acc r = ident;
#pragma unroll
                    for (int j = 0; j < ITEMS; ++j) {
                        Acc x[EG];
                        load_chunk(sm, chunk_of(sub, j), t0, lo, hi, x);
                        Acc c = x[0];
#pragma unroll
                        for (int k = 1; k < EG; ++k)
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

    __device__ __forceinline__ static uint4 *plane(Smem &sm, int p, int c) {
        return p == 0 ? &sm.stage[c] : &sm.extra[(p - 1) * kChunks + c];
    }
    __device__ __forceinline__ static void put(Smem &sm, int gi, const Acc (&x)[EG]) {
#pragma unroll
        for (int q = 0; q < V; ++q) {
            const int c = gi * V + q;
#pragma unroll
            for (int p = 0; p < kPlanes; ++p) {
                uint4 w;
                Acc *d = reinterpret_cast<Acc *>(&w);
#pragma unroll
                for (int r = 0; r < kPerPlane; ++r)
                    d[r] = (p * kPerPlane + r < E) ? x[q * E + p * kPerPlane + r] : Acc(0);
                *plane(sm, p, c) = w;
            }
        }
    }
    __device__ __forceinline__ static void get(Smem &sm, int gi, Acc (&x)[EG]) {
#pragma unroll
        for (int q = 0; q < V; ++q) {
            const int c = gi * V + q;
#pragma unroll
            for (int p = 0; p < kPlanes; ++p) {
                const uint4 w = *plane(sm, p, c);
                const Acc *d = reinterpret_cast<const Acc *>(&w);
#pragma unroll
                for (int r = 0; r < kPerPlane; ++r)
                    if (p * kPerPlane + r < E)
                        x[q * E + p * kPerPlane + r] = d[r];
            }
        }
    }
    // Store a group's outputs: 16-byte stores for whole aligned chunks.
    __device__ __forceinline__ static void store_group(S *eout, bool aligned_io, int64_t v, int64_t lo,
                                                       int64_t hi, const Acc (&x)[EG]) {
#pragma unroll
        for (int q = 0; q < V; ++q) {
            const int64_t vq = v + q * E;
            Acc part[E];
#pragma unroll
            for (int k = 0; k < E; ++k)
                part[k] = x[q * E + k];
            if (aligned_io && vq >= lo && vq + E <= hi) {
                st_v4(reinterpret_cast<uint4 *>(eout) + vq / E, C::pack(part));
            } else if (vq < hi && vq + E > lo) {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (vq + k >= lo && vq + k < hi)
                        C::store1(eout + vq + k, part[k]);
            }
        }
    }
};

template <class S, class Op, int ITEMS, int SUB, int THREADS, int V>
__global__ void __launch_bounds__(THREADS) k_scan_staged(SegArgs a) {
    using G = Staged<S, Op, ITEMS, SUB, THREADS, V>;
    using Acc = typename G::Acc;
    using C = typename G::C;
    constexpr int E = G::E;
    constexpr int EG = G::EG;
    extern __shared__ __align__(128) unsigned char dsm[];
    typename G::Smem &sm = *reinterpret_cast<typename G::Smem *>(dsm);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const Acc ident = Op::template identity<Acc>();
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
            const uint32_t bytes = (uint32_t)((cend - c0) * 16);
            mbar_arrive_expect_tx(&sm.bar, bytes);
            bulk_g2s(&sm.stage[0], vin + c0, bytes, &sm.bar);
        }
        const bool ok = mbar_wait(&sm.bar, phase, kCopyWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0)
                atomicCAS(&g_mt_err, 0, kErrTimeout);
            mbar_wait(&sm.bar, phase, kCopyWaitLimit);  // drain the copy before leaving
            return;
        }
        phase ^= 1u;

        // Pass 0: the super-tile's aggregate, published before the scan so
        // that later tiles' look-backs find it as early as possible.
        const Acc agg_total = G::reduce(sm, t0, lo, hi);
        publish_aggregate<Acc, Op>(a.lb, g, first, agg_total);
#if MT_STAGED_EARLY_LOOKBACK
        // The prefix right away; the scan below then stores final outputs.
        const Acc tp = lookback_prefix<Acc, Op>(a.lb, g, first, agg_total, &sm.prefix[it & 1]);
#endif

        // Pass 1: scan the sub-tiles in order with a running carry; keep each
        // element's super-tile-local prefix in shared memory.
        Acc carry = ident;
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
            Acc x[ITEMS][EG];
#pragma unroll
            for (int j = 0; j < ITEMS; ++j)
                G::load_chunk(sm, G::chunk_of(sub, j), t0, lo, hi, x[j]);
            Acc inc[ITEMS];
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
#pragma unroll
                for (int k = 1; k < EG; ++k)
                    x[j][k] = Op::apply(x[j][k - 1], x[j][k]);
                inc[j] = x[j][EG - 1];
            }
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
                for (int j = 0; j < ITEMS; ++j) {
                    const Acc y = __shfl_up_sync(kFull, inc[j], d);
                    if (lane >= d)
                        inc[j] = Op::apply(y, inc[j]);
                }
            }
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
                sm.warp_tot[sub & 1][warp] = run;
            __syncthreads();
            Acc wpre = ident, agg = ident;
#pragma unroll
            for (int w = 0; w < G::kNW; ++w) {
                const Acc t = sm.warp_tot[sub & 1][w];
                if (w < warp)
                    wpre = Op::apply(wpre, t);
                agg = Op::apply(agg, t);
            }
#if MT_STAGED_EARLY_LOOKBACK
            const Acc base0 = Op::apply(Op::apply(tp, carry), wpre);
#else
            const Acc base0 = Op::apply(carry, wpre);
#endif
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const Acc base = Op::apply(base0, pre[j]);
                if (a.inclusive) {
#pragma unroll
                    for (int k = 0; k < EG; ++k)
                        x[j][k] = Op::apply(base, x[j][k]);
                } else {
#pragma unroll
                    for (int k = EG - 1; k > 0; --k)
                        x[j][k] = Op::apply(base, x[j][k - 1]);
                    x[j][0] = base;
                }
                const int gi = G::chunk_of(sub, j);
                const int64_t v = t0 + (int64_t)gi * EG;
#if MT_STAGED_EARLY_LOOKBACK
                G::store_group(eout, a.aligned_io != 0, v, lo, hi, x[j]);
#else
                if (v < hi && v + EG > lo)
                    G::put(sm, gi, x[j]);
#endif
            }
            carry = Op::apply(carry, agg);
        }
#if !MT_STAGED_EARLY_LOOKBACK

        // The super-tile's prefix (publishes its aggregate, looks back, and
        // publishes its inclusive prefix; identity for a segment's first one).
        const Acc tp = lookback_prefix<Acc, Op>(a.lb, g, first, agg_total, &sm.prefix[it & 1]);

        // Pass 2: prefix + local prefix, narrowed to S and stored.
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll
            for (int j = 0; j < ITEMS; ++j) {
                const int gi = G::chunk_of(sub, j);
                const int64_t v = t0 + (int64_t)gi * EG;
                if (!(v < hi && v + EG > lo))
                    continue;
                Acc x[EG];
                G::get(sm, gi, x);
#pragma unroll
                for (int k = 0; k < EG; ++k)
                    x[k] = Op::apply(tp, x[k]);
                G::store_group(eout, a.aligned_io != 0, v, lo, hi, x);
            }
        }
#endif
        fence_proxy_async_smem();  // this thread's shared writes precede the next bulk copy
    }
}

template <class S, class Op, int ITEMS, int SUB, int THREADS, int V = 1>
static cudaError_t launch_staged(const SegArgs &a, int64_t max_ctas, const Launch &L) {
    using G = Staged<S, Op, ITEMS, SUB, THREADS, V>;
    static int per_sm[128] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        e = cudaFuncSetAttribute(k_scan_staged<S, Op, ITEMS, SUB, THREADS, V>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        // the whole unified L1/shared array as shared memory, so that as many
        // super-tiles as registers allow are in flight on each SM
        e = cudaFuncSetAttribute(k_scan_staged<S, Op, ITEMS, SUB, THREADS, V>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_scan_staged<S, Op, ITEMS, SUB, THREADS, V>,
                                                          THREADS, G::kSmemBytes);
        if (e != cudaSuccess)
            return e;
        per_sm[dev] = b > 0 ? b : 1;
    }
    int64_t grid = (int64_t)L.sm_count * per_sm[dev];
    if (max_ctas > 0 && grid > max_ctas)
        grid = max_ctas;
    if (grid < 1)
        grid = 1;
    k_scan_staged<S, Op, ITEMS, SUB, THREADS, V><<<(unsigned)grid, THREADS, G::kSmemBytes, L.stream>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace mt
