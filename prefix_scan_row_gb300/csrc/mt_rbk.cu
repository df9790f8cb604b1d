// mt_rbk.cu -- reduce by key: every run of consecutive equal keys becomes one
// output entry (key, sum of the run's values), in input order.
//
// Semantics follow the Quadrants "Algorithms" user guide, section
// "qd.algorithms.reduce_by_key_add": keys and values are i32, u32 or f32;
// keys equal but separated by other keys form separate runs; num_runs gets
// the number of runs and only the first num_runs output entries are written.
// Float keys compare with ==, so each NaN is a run of its own and -0 equals
// +0 (the run keeps the key of its first element).
//
// The page realises it as a head-flag pass, a scan of the flags, a zeroing
// pass and an atomic scatter. Here one persistent kernel reads keys and
// values once: each element carries the pair (h, v) -- h = 1 when it starts a
// run -- and the tile scans pairs with the segmented operator
//   (c1, s1) + (c2, s2) = (c1 + c2, c2 != 0 ? s2 : s1 + s2),
// whose inclusive prefix at an element is (runs started so far, sum of the
// open run). Super-tiles of 4096 keys and values arrive in shared memory by
// bulk copies. A first pass over the 16-byte chunks (consecutive lanes,
// consecutive chunks: no bank conflicts) finds each chunk's head bits and its
// own pair; each thread then folds the pairs of 4 consecutive chunks, so one
// pair per thread enters the warp and block scans; the super-tile's own pair
// is published as soon as that scan is done; warp 0 then looks back for the
// pairs of all earlier super-tiles (packed in 64 bits); every chunk's prefix
// goes back to shared memory, and a second chunk pass writes the results:
// heads keys_out[c - 1], run ends values_out[c - 1]. No atomics
// on the outputs, and sums are added in a fixed order.
#include <cstddef>
#include <type_traits>

#include "mt_lookback.cuh"

namespace mt {

#ifndef MT_RBK_TILE
#define MT_RBK_TILE 4096  // elements per super-tile: 4096 or 8192
#endif
#ifndef MT_RBK_THREADS
#define MT_RBK_THREADS 256
#endif
constexpr int kRbkThreads = MT_RBK_THREADS;
constexpr int kRbkSeg = 16;                                       // consecutive elements per thread segment
constexpr int kRbkSub = MT_RBK_TILE / (kRbkThreads * kRbkSeg);    // segments per thread per super-tile
static_assert(kRbkSub >= 1 && kRbkSub * kRbkThreads * kRbkSeg == MT_RBK_TILE, "super-tile shape");
constexpr int kRbkSubElems = kRbkThreads * kRbkSeg;               // elements per sub-tile (4096)
constexpr int64_t kRbkTE = (int64_t)kRbkSub * kRbkSubElems;       // elements per super-tile (4096)
constexpr int kRbkChunks = (int)(kRbkTE / 4);                     // 16-byte chunks per super-tile

struct RbkArgs {
    const char *keys;   // keys and values share their 16-byte phase
    const char *vals;
    uint32_t *keys_out;
    uint32_t *vals_out;
    int32_t *num_runs;
    const int32_t *n_dev;
    unsigned long long *counter;
    LookBack lb;
};

// The pair (c, s) packed as c << 32 | bits(s); VF: s is an f32, else a
// wrapping 32-bit integer sum.
template <bool VF>
struct SegOp {
    template <class T> __device__ __forceinline__ static T identity() { return T(0); }
    __device__ __forceinline__ static uint64_t apply(uint64_t a, uint64_t b) {
        const uint32_t cb = (uint32_t)(b >> 32);
        const uint32_t ca = (uint32_t)(a >> 32);
        uint32_t s;
        if (cb != 0u)
            s = (uint32_t)b;
        else if (VF)
            s = __float_as_uint(__uint_as_float((uint32_t)a) + __uint_as_float((uint32_t)b));
        else
            s = (uint32_t)a + (uint32_t)b;
        return ((uint64_t)(ca + cb) << 32) | s;
    }
};

// The same pair unpacked, for the scan inside a tile: c counts heads, s is
// an f32 (VF) or a wrapping u32 sum.
template <bool VF>
struct Seg {
    using V = typename std::conditional<VF, float, uint32_t>::type;
    uint32_t c;
    V s;
    __device__ __forceinline__ static Seg ident() { return Seg{0u, V(0)}; }
    __device__ __forceinline__ static Seg apply(const Seg &a, const Seg &b) {
        return Seg{a.c + b.c, b.c != 0u ? b.s : a.s + b.s};
    }
    __device__ __forceinline__ static V val(uint32_t bits) {
        if constexpr (VF)
            return __uint_as_float(bits);
        else
            return bits;
    }
    __device__ __forceinline__ static uint32_t bits(V v) {
        if constexpr (VF)
            return __float_as_uint(v);
        else
            return v;
    }
    __device__ __forceinline__ static Seg unpack(uint64_t p) { return Seg{(uint32_t)(p >> 32), val((uint32_t)p)}; }
    __device__ __forceinline__ Seg shfl_up(int d) const {
        return Seg{__shfl_up_sync(kFull, c, d), __shfl_up_sync(kFull, s, d)};
    }
    __device__ __forceinline__ Seg shfl(int l) const {
        return Seg{__shfl_sync(kFull, c, l), __shfl_sync(kFull, s, l)};
    }
};

template <bool KF>
__device__ __forceinline__ bool keys_differ(uint32_t a, uint32_t b) {
    if (KF)
        return __uint_as_float(a) != __uint_as_float(b);  // NaN differs from everything
    return a != b;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Shared state of one CTA: the super-tile's keys and values (bulk-copied),
// the keys just before and after it, and the block's scratch.
struct RbkSmem {
    uint4 keys[kRbkChunks];
    uint4 vals[kRbkChunks];
    uint32_t csum[kRbkChunks]; // per chunk: its own open-run sum, then the sum part of its prefix
    uint32_t ccnt[kRbkChunks]; // per chunk: the count part of its prefix
    uint8_t heads[kRbkChunks]; // head bits of each chunk (bit k: its element k)
    uint64_t bar;
    unsigned long long tile;
    uint32_t kprev, knext;     // the neighbours' keys (when they exist)
    uint32_t warp_c[kRbkSub][kRbkThreads / 32];  // warp totals of the segment scan
    uint32_t warp_s[kRbkSub][kRbkThreads / 32];
    uint32_t wex_c[kRbkSub][kRbkThreads / 32];   // and the warps' exclusive prefixes
    uint32_t wex_s[kRbkSub][kRbkThreads / 32];
    uint64_t prefix;
};
// csum and ccnt are read and written 16 bytes at a time, heads 4 at a time
static_assert(offsetof(RbkSmem, csum) % 16 == 0 && offsetof(RbkSmem, ccnt) % 16 == 0 &&
                  offsetof(RbkSmem, heads) % 4 == 0 && offsetof(RbkSmem, bar) % 8 == 0,
              "shared-memory layout of the reduce-by-key kernel");

// One staged super-tile: valid elements [llo, lhi) ([0, kRbkTE) when FULL);
// has_first: it holds the first element (a head whatever its key); has_last:
// it holds the last one (which ends its run and gives num_runs).
// n_live bounds every output index: a valid run index always lies below it,
// and a prefix left incomplete by a look-back that gave up (the error word is
// set then) must not send a write outside the outputs.
template <bool KF, bool VF, bool FULL>
__device__ __forceinline__ void rbk_tile(RbkSmem &sm, const RbkArgs &a, int64_t g, int llo, int lhi,
                                         bool has_first, bool has_last, uint32_t n_live) {
    using P = Seg<VF>;
    using Op = SegOp<VF>;
    using St = Status<uint64_t>;
    constexpr int kNW = kRbkThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t *skey = reinterpret_cast<const uint32_t *>(sm.keys);
    const uint32_t kprev = sm.kprev, knext = sm.knext;

    // Pass A, chunk by chunk (consecutive lanes, consecutive 16-byte chunks:
    // no bank conflicts): head bits and the sum of the chunk's open run. The
    // key before a chunk is the last key of the lane to the left.
#pragma unroll 1
    for (int c = threadIdx.x; c < kRbkChunks; c += kRbkThreads) {
        const uint4 kk = lds128(&sm.keys[c]);
        const uint4 vv4 = lds128(&sm.vals[c]);
        uint32_t prev = __shfl_up_sync(kFull, kk.w, 1);
        if (lane == 0)
            prev = (4 * c - 1 >= llo) ? skey[4 * c - 1] : kprev;
        uint32_t m = 0u;
        typename P::V sum = typename P::V(0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = 4 * c + k;
            const uint32_t key = word(kk, k);
            if (FULL || (i >= llo && i < lhi)) {
                // the first element starts a run whatever its key
                const bool first = has_first && (FULL ? (k == 0 && c == 0) : i == llo);
                const bool h = first || keys_differ<KF>(key, prev);
                m |= (h ? 1u : 0u) << k;
                const typename P::V v = P::val(word(vv4, k));
                sum = h ? v : sum + v;
            }
            prev = key;
        }
        sm.heads[c] = (uint8_t)m;
        sm.csum[c] = P::bits(sum);
    }
    __syncthreads();

    // Each thread owns segments of 4 consecutive chunks (16 elements): their
    // pairs from the chunk pairs, in order.
    P seg[kRbkSub], cpre[kRbkSub][4];
#pragma unroll
    for (int sub = 0; sub < kRbkSub; ++sub) {
        const int c0 = 4 * (sub * kRbkThreads + threadIdx.x);
        const uint32_t m4 = *reinterpret_cast<const uint32_t *>(&sm.heads[c0]);
        const uint4 s4 = lds128(reinterpret_cast<const uint4 *>(&sm.csum[c0]));
        P acc = P::ident();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            cpre[sub][q] = acc;
            acc = P::apply(acc, P{(uint32_t)__popc((m4 >> (8 * q)) & 0xffu), P::val(word(s4, q))});
        }
        seg[sub] = acc;
    }

    // The segments' exclusive prefixes in order (sub-tile, then thread):
    // warp scans; warp 0 scans the warp totals.
    P ex[kRbkSub];
#pragma unroll
    for (int sub = 0; sub < kRbkSub; ++sub) {
        P inc = seg[sub];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const P y = inc.shfl_up(d);
            if (lane >= d)
                inc = P::apply(y, inc);
        }
        P e = inc.shfl_up(1);
        if (lane == 0)
            e = P::ident();
        ex[sub] = e;
        if (lane == 31) {
            sm.warp_c[sub][warp] = inc.c;
            sm.warp_s[sub][warp] = P::bits(inc.s);
        }
    }
    __syncthreads();  // warp totals are written

    // Warp 0: the warps' exclusive prefixes, the super-tile's pair (published
    // at once), the look-back, the inclusive prefix.
    if (warp == 0) {
        P agg = P::ident();
#pragma unroll
        for (int sub = 0; sub < kRbkSub; ++sub) {
            P w = lane < kNW ? P{sm.warp_c[sub][lane], P::val(sm.warp_s[sub][lane])} : P::ident();
#pragma unroll
            for (int d = 1; d < kNW; d <<= 1) {
                const P y = w.shfl_up(d);
                if (lane >= d)
                    w = P::apply(y, w);
            }
            P we = w.shfl_up(1);
            if (lane == 0)
                we = P::ident();
            const P tot = w.shfl(kNW - 1);
            if (lane < kNW) {
                const P before = P::apply(agg, we);
                sm.wex_c[sub][lane] = before.c;
                sm.wex_s[sub][lane] = P::bits(before.s);
            }
            agg = P::apply(agg, tot);
        }
        const uint64_t aggp = ((uint64_t)agg.c << 32) | P::bits(agg.s);
        publish_aggregate<uint64_t, Op>(a.lb, g, 0, aggp);
        uint64_t pre = 0;  // the identity pair
        if (a.lb.recs != nullptr && g != 0) {
            pre = warp_lookback<uint64_t, Op>(a.lb.recs, g, 0, a.lb.spin_limit);
            if (lane == 0 && g != a.lb.skip_tile)
                St::publish(a.lb.recs + g * St::kSlots, kIncl, Op::apply(pre, aggp));
        }
        if (lane == 0)
            sm.prefix = pre;
    }
    __syncthreads();

    // Every chunk's prefix, written back by the segment's owner.
    const P tp = P::unpack(sm.prefix);
#pragma unroll
    for (int sub = 0; sub < kRbkSub; ++sub) {
        const int c0 = 4 * (sub * kRbkThreads + threadIdx.x);
        const P base = P::apply(P::apply(tp, P{sm.wex_c[sub][warp], P::val(sm.wex_s[sub][warp])}), ex[sub]);
        const P q0 = P::apply(base, cpre[sub][0]), q1 = P::apply(base, cpre[sub][1]);
        const P q2 = P::apply(base, cpre[sub][2]), q3 = P::apply(base, cpre[sub][3]);
        sts128(reinterpret_cast<uint4 *>(&sm.csum[c0]),
               make_uint4(P::bits(q0.s), P::bits(q1.s), P::bits(q2.s), P::bits(q3.s)));
        sts128(reinterpret_cast<uint4 *>(&sm.ccnt[c0]), make_uint4(q0.c, q1.c, q2.c, q3.c));
    }
    // Does the super-tile's last element end its run?
    const bool last_ends = lhi > llo && (has_last || keys_differ<KF>(knext, skey[lhi - 1]));
    const int c_last = (lhi - 1) >> 2;  // the chunk of the last valid element
    __syncthreads();

    // Pass B, chunk by chunk again: heads write their key, run ends the
    // run's sum, at run index c - 1.
#pragma unroll 1
    for (int c = threadIdx.x; c < kRbkChunks; c += kRbkThreads) {
        const uint32_t m = sm.heads[c];
        uint32_t e;  // element k ends a run: k + 1 starts one, or k is the last
        if (FULL) {
            const uint32_t mn = (c + 1 < kRbkChunks) ? sm.heads[c + 1] : (last_ends ? 1u : 0u);
            e = (m >> 1) | ((mn & 1u) << 3);
        } else {
            const uint32_t mn = (c + 1 < kRbkChunks) ? sm.heads[c + 1] : 0u;
            e = (m >> 1) | ((mn & 1u) << 3);
            const int li = lhi - 1 - 4 * c;
            if (li >= 0 && li < 4)
                e = (e & ((1u << li) - 1u)) | ((last_ends ? 1u : 0u) << li);
            else if (li < 0)
                e = 0u;
            const int lv = llo - 4 * c;  // elements before the first valid one end nothing
            if (lv > 0)
                e &= lv >= 4 ? 0u : ~((1u << lv) - 1u);
        }
        const uint4 vv4 = lds128(&sm.vals[c]);
        const uint4 kk = lds128(&sm.keys[c]);
        P run{sm.ccnt[c], P::val(sm.csum[c])};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = 4 * c + k;
            const bool h = (m >> k) & 1u;
            if (FULL || (i >= llo && i < lhi)) {
                run.c += h ? 1u : 0u;
                run.s = h ? P::val(word(vv4, k)) : run.s + P::val(word(vv4, k));
            }
            const uint32_t r = run.c - 1u;
            if (h && r < n_live)
                a.keys_out[r] = word(kk, k);
            if (((e >> k) & 1u) && r < n_live)
                a.vals_out[r] = P::bits(run.s);
        }
        if (has_last && c == c_last)
            *a.num_runs = (int32_t)(run.c <= n_live ? run.c : n_live);
    }
}

template <bool KF, bool VF>
__global__ void __launch_bounds__(kRbkThreads) k_reduce_by_key(RbkArgs a) {
    pdl_prologue();
    extern __shared__ __align__(128) unsigned char dsm[];
    RbkSmem &sm = *reinterpret_cast<RbkSmem *>(dsm);

    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t head = (int64_t)(((uintptr_t)a.keys & 15u) / 4);
    const uint4 *vk = reinterpret_cast<const uint4 *>(a.keys - head * 4);
    const uint4 *vv = reinterpret_cast<const uint4 *>(a.vals - head * 4);
    const uint32_t *ek = reinterpret_cast<const uint32_t *>(a.keys) - head;  // virtual element 0
    const int64_t lo = head, hi = head + n;
    const int64_t ntiles = n > 0 ? (hi + kRbkTE - 1) / kRbkTE : 0;

    if (threadIdx.x == 0) {
        mbar_init(&sm.bar, 1);
        fence_mbar_init();
    }
    uint32_t phase = 0;
    for (int64_t it = 0;; ++it) {
        if (threadIdx.x == 0)
            sm.tile = atomicAdd(a.counter, 1ull);
        __syncthreads();  // tile id visible; every thread is done with the last super-tile
        const int64_t g = (int64_t)sm.tile;
        if (g >= ntiles)
            break;
        const int64_t t0 = g * kRbkTE;
        // in-tile valid range [llo, lhi) of virtual elements
        const int llo = lo > t0 ? (int)(lo - t0) : 0;
        const int lhi = hi - t0 < kRbkTE ? (int)(hi - t0) : (int)kRbkTE;
        if (threadIdx.x == 0) {
            fence_proxy_async_smem();  // the last iteration's shared accesses come first
            const int64_t c0 = t0 / 4;
            int64_t cend = (hi + 3) / 4;
            if (cend > c0 + kRbkChunks)
                cend = c0 + kRbkChunks;
            const uint32_t bytes = (uint32_t)((cend - c0) * 16);
            mbar_arrive_expect_tx(&sm.bar, 2 * bytes);
            bulk_g2s(&sm.keys[0], vk + c0, bytes, &sm.bar);
            bulk_g2s(&sm.vals[0], vv + c0, bytes, &sm.bar);
            sm.kprev = (t0 + llo - 1 >= lo) ? __ldg(ek + t0 + llo - 1) : 0u;
            sm.knext = (t0 + lhi < hi) ? __ldg(ek + t0 + lhi) : 0u;
        }
        bool ok = true;
        if (threadIdx.x < 32)
            ok = mbar_wait(&sm.bar, phase, kCopyWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) {
                atomicCAS(&g_mt_err, 0, kErrTimeout);
                mbar_wait(&sm.bar, phase, kCopyWaitLimit);  // drain the copies before leaving
            }
            return;
        }
        phase ^= 1u;
        if (llo == 0 && lhi == (int)kRbkTE)
            rbk_tile<KF, VF, true>(sm, a, g, 0, (int)kRbkTE, g == 0, t0 + kRbkTE == hi, (uint32_t)n);
        else
            rbk_tile<KF, VF, false>(sm, a, g, llo, lhi, g == 0, t0 + lhi == hi, (uint32_t)n);
        fence_proxy_async_smem();  // this thread's shared accesses precede the next bulk copies
    }
}

template <bool KF, bool VF>
static cudaError_t launch_rbk(const RbkArgs &a, const Launch &L) {
    static PerDevice per_sm;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int bytes = (int)sizeof(RbkSmem);
    int blocks = per_sm.get(dev);
    if (blocks == 0) {
        e = cudaFuncSetAttribute(k_reduce_by_key<KF, VF>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess)
            return e;
        e = cudaFuncSetAttribute(k_reduce_by_key<KF, VF>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return e;
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_reduce_by_key<KF, VF>, kRbkThreads, bytes);
        if (e != cudaSuccess)
            return e;
        blocks = b > 0 ? b : 1;
        per_sm.set(dev, blocks);
    }
    e = launch_pdl(k_reduce_by_key<KF, VF>, (unsigned)(L.sm_count * blocks), kRbkThreads, bytes,
                   L.stream, a);
    note_launch();
    return e;
}

int64_t rbk_tile_elems() { return kRbkTE; }
int rbk_rec_slots() { return Status<uint64_t>::kSlots; }

cudaError_t rbk_launch(const void *keys, const void *vals, void *keys_out, void *vals_out, int32_t *num_runs,
                       uint64_t *scratch, const int32_t *n_dev, bool key_float, bool val_float,
                       const Launch &L) {
    RbkArgs a;
    a.keys = static_cast<const char *>(keys);
    a.vals = static_cast<const char *>(vals);
    a.keys_out = static_cast<uint32_t *>(keys_out);
    a.vals_out = static_cast<uint32_t *>(vals_out);
    a.num_runs = num_runs;
    a.n_dev = n_dev;
    a.counter = reinterpret_cast<unsigned long long *>(scratch);
    a.lb.recs = scratch + kHeaderSlots;
    a.lb.skip_tile = L.skip_tile;
    a.lb.spin_limit = L.spin_limit;
    if (key_float)
        return val_float ? launch_rbk<true, true>(a, L) : launch_rbk<true, false>(a, L);
    return val_float ? launch_rbk<false, true>(a, L) : launch_rbk<false, false>(a, L);
}

cudaError_t rbk_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
