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
// open run). Super-tiles of 6144 keys and values arrive in shared memory by
// bulk copies. Each thread owns units of 8 consecutive elements (two 16-byte
// chunks, read in an order that keeps shared memory free of bank conflicts):
// a first pass finds each unit's head bits and its pair, warp scans and a
// scan of the warp totals give every unit its prefix inside the super-tile,
// the super-tile's pair is published at once, and warp 0 looks back for the
// pairs of all earlier super-tiles (packed in 64 bits). A second pass over
// the units writes the results: heads keys_out[c - 1], run ends
// values_out[c - 1]. No atomics
// on the outputs, and sums are added in a fixed order.
#include <cstddef>
#include <type_traits>

#include "mt_lookback.cuh"

namespace mt {

#ifndef MT_RBK_LB_PER_LANE
#define MT_RBK_LB_PER_LANE 1  // predecessors per lane per look-back poll
#endif
constexpr int kRbkLbPerLane = MT_RBK_LB_PER_LANE;
#ifndef MT_RBK_EARLY
#define MT_RBK_EARLY 1  // publish each super-tile's pair from a keys-only pass, before the scan
#endif
#ifndef MT_RBK_TILE
#define MT_RBK_TILE 6144  // elements per super-tile (a multiple of 2048)
#endif
constexpr int kRbkThreads = 256;
constexpr int kRbkUnitElems = 8;                                  // a unit: two adjacent 16-byte chunks
constexpr int kRbkSub = MT_RBK_TILE / (kRbkThreads * kRbkUnitElems);  // units per thread per super-tile
static_assert(kRbkSub >= 1 && kRbkSub * kRbkThreads * kRbkUnitElems == MT_RBK_TILE, "super-tile shape");
constexpr int64_t kRbkTE = MT_RBK_TILE;                           // elements per super-tile
constexpr int kRbkChunks = (int)(kRbkTE / 4);                     // 16-byte chunks per super-tile
constexpr int kRbkUnits = (int)(kRbkTE / kRbkUnitElems);          // units per super-tile

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
// the keys just before and after it, each unit's head bits, and the block's
// scratch.
struct RbkSmem {
    uint4 keys[kRbkChunks];
    uint4 vals[kRbkChunks];
    uint8_t heads[kRbkUnits];  // head bits of each unit (bit k: its element k)
    uint64_t bar;
    unsigned long long tile;
    uint32_t kprev, knext;     // the neighbours' keys (when they exist)
    uint32_t warp_c[kRbkSub][kRbkThreads / 32];  // warp totals of each sub-tile's scan
    uint32_t warp_s[kRbkSub][kRbkThreads / 32];
    uint32_t hcount[kRbkThreads / 32];  // each warp's heads in the super-tile
    int32_t hlast[kRbkThreads / 32];    // each warp's last head (-1: none)
    uint64_t agg;                       // the super-tile's pair
    uint64_t prefix;
};
static_assert(offsetof(RbkSmem, bar) % 8 == 0, "shared-memory layout of the reduce-by-key kernel");

// Unit u (chunks 2u and 2u + 1) of a staged array. Lanes 4-7 of every group
// of 8 read the second chunk first, so the 8 lanes that share a wavefront
// touch 8 different 16-byte bank groups.
__device__ __forceinline__ void load_unit(const uint4 *base, int u, uint4 &c0, uint4 &c1) {
    const bool sw = (threadIdx.x >> 2) & 1;
    const bool in = MT_CHECK_INDEX(2 * u, kRbkChunks) && MT_CHECK_INDEX(2 * u + 1, kRbkChunks);
    const uint4 p = in ? lds128(&base[2 * u + (sw ? 1 : 0)]) : make_uint4(0u, 0u, 0u, 0u);
    const uint4 q = in ? lds128(&base[2 * u + (sw ? 0 : 1)]) : make_uint4(0u, 0u, 0u, 0u);
    c0 = sw ? q : p;
    c1 = sw ? p : q;
}
__device__ __forceinline__ uint32_t word8(const uint4 &c0, const uint4 &c1, int k) {
    return k < 4 ? word(c0, k) : word(c1, k - 4);
}

// One staged super-tile: valid elements [llo, lhi) ([0, kRbkTE) when FULL);
// has_first: it holds the first element (a head whatever its key); has_last:
// it holds the last one (which ends its run and gives num_runs). n_live
// bounds every output index: a valid run index always lies below it, and a
// prefix left incomplete by a look-back that gave up (the error word is set
// then) must not send a write outside the outputs.
//
// Thread t owns unit s * 256 + t of sub-tile s. Pass 1 finds each unit's
// head bits and its pair (heads, sum of the open run), and scans the pairs
// (warps by shuffles, then the warp totals across lanes, sub-tiles in
// order); warp 0 publishes the super-tile's pair and looks back. Pass 2
// reads each unit again and writes its outputs from the unit's full prefix.
template <bool KF, bool VF, bool FULL>
__device__ __forceinline__ void rbk_tile(RbkSmem &sm, const RbkArgs &a, int64_t g, int llo, int lhi,
                                         bool has_first, bool has_last, uint32_t n_live) {
    using P = Seg<VF>;
    using V = typename P::V;
    using Op = SegOp<VF>;
    constexpr int kNW = kRbkThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t *skey = reinterpret_cast<const uint32_t *>(sm.keys);
    const uint32_t kprev = sm.kprev, knext = sm.knext;

    uint32_t mh[kRbkSub];
#if MT_RBK_EARLY
    // Pass 0: each unit's head bits from the keys alone (the key before a
    // unit is the last key of the lane to the left), and the super-tile's
    // head count and last head.
    {
        uint32_t cnt = 0u;
        int last = -1;
#pragma unroll
        for (int s = 0; s < kRbkSub; ++s) {
            const int u = s * kRbkThreads + threadIdx.x;
            uint4 k0, k1;
            load_unit(sm.keys, u, k0, k1);
            uint32_t prev = __shfl_up_sync(kFull, k1.w, 1);
            if (lane == 0)
                prev = (8 * u - 1 >= llo && MT_CHECK_INDEX(8 * u - 1, kRbkTE)) ? skey[8 * u - 1] : kprev;
            uint32_t m = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 8 * u + k;
                const uint32_t key = word8(k0, k1, k);
                if (FULL || (i >= llo && i < lhi)) {
                    // the first element starts a run whatever its key
                    const bool first = has_first && (FULL ? (k == 0 && u == 0) : i == llo);
                    m |= ((first || keys_differ<KF>(key, prev)) ? 1u : 0u) << k;
                }
                prev = key;
            }
            if (MT_CHECK_INDEX(u, kRbkUnits))
                sm.heads[u] = (uint8_t)m;
            mh[s] = m;
            cnt += (uint32_t)__popc(m);
            if (m != 0u)
                last = 8 * u + 31 - __clz(m);  // units grow with s: the thread's last head
        }
        cnt = __reduce_add_sync(kFull, cnt);
        last = __reduce_max_sync(kFull, last);
        if (lane == 0) {
            sm.hcount[warp] = cnt;
            sm.hlast[warp] = last;
        }
    }
    __syncthreads();  // head bits and per-warp counts are written
    // The last warp publishes the super-tile's pair before the scan: the
    // head count, and the sum of the values from the last head on (of all
    // valid values when the tile has no head), so later tiles' look-backs
    // find it sooner.
    if (warp == kNW - 1) {
        const uint32_t c = __reduce_add_sync(kFull, lane < kNW ? sm.hcount[lane] : 0u);
        const int hl = __reduce_max_sync(kFull, lane < kNW ? sm.hlast[lane] : -1);
        const uint32_t *sval = reinterpret_cast<const uint32_t *>(sm.vals);
        V part = V(0);
        for (int i = (hl >= 0 ? hl : llo) + lane; i < lhi; i += 32)
            part += P::val(MT_CHECK_INDEX(i, kRbkTE) ? sval[i] : 0u);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1)
            part += __shfl_xor_sync(kFull, part, d);
        if (lane == 0) {
            const uint64_t aggp = ((uint64_t)c << 32) | P::bits(part);
            sm.agg = aggp;
            if (a.lb.recs != nullptr && g != a.lb.skip_tile)
                publish_record<uint64_t>(a.lb, g, g == 0 ? kIncl : kAgg, aggp);
        }
    }
#endif

    // Pass 1. The key before a unit is the last key of the lane to the left.
    P ex[kRbkSub];
#pragma unroll
    for (int s = 0; s < kRbkSub; ++s) {
        const int u = s * kRbkThreads + threadIdx.x;
        uint4 v0, v1;
        load_unit(sm.vals, u, v0, v1);
#if MT_RBK_EARLY
        const uint32_t m = mh[s];
        V sum = V(0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = 8 * u + k;
            if (FULL || (i >= llo && i < lhi)) {
                const V v = P::val(word8(v0, v1, k));
                sum = ((m >> k) & 1u) ? v : sum + v;
            }
        }
#else
        uint4 k0, k1;
        load_unit(sm.keys, u, k0, k1);
        uint32_t prev = __shfl_up_sync(kFull, k1.w, 1);
        if (lane == 0)
            prev = (8 * u - 1 >= llo && MT_CHECK_INDEX(8 * u - 1, kRbkTE)) ? skey[8 * u - 1] : kprev;
        uint32_t m = 0u;
        V sum = V(0);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = 8 * u + k;
            const uint32_t key = word8(k0, k1, k);
            if (FULL || (i >= llo && i < lhi)) {
                // the first element starts a run whatever its key
                const bool first = has_first && (FULL ? (k == 0 && u == 0) : i == llo);
                const bool h = first || keys_differ<KF>(key, prev);
                m |= (h ? 1u : 0u) << k;
                const V v = P::val(word8(v0, v1, k));
                sum = h ? v : sum + v;
            }
            prev = key;
        }
        if (MT_CHECK_INDEX(u, kRbkUnits))
            sm.heads[u] = (uint8_t)m;
        mh[s] = m;
#endif
        P inc{(uint32_t)__popc(m), sum};
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const P y = inc.shfl_up(d);
            if (lane >= d)
                inc = P::apply(y, inc);
        }
        P e = inc.shfl_up(1);
        if (lane == 0)
            e = P::ident();
        ex[s] = e;
        if (lane == 31) {
            sm.warp_c[s][warp] = inc.c;
            sm.warp_s[s][warp] = P::bits(inc.s);
        }
    }
    __syncthreads();  // warp totals and head bits are written

    // Each unit's prefix inside the super-tile: the warp totals of each
    // sub-tile scanned across the first kNW lanes, sub-tiles in order.
    P base[kRbkSub];
    P carry = P::ident();
#pragma unroll
    for (int s = 0; s < kRbkSub; ++s) {
        P t = lane < kNW ? P{sm.warp_c[s][lane], P::val(sm.warp_s[s][lane])} : P::ident();
#pragma unroll
        for (int d = 1; d < kNW; d <<= 1) {
            const P y = t.shfl_up(d);
            if (lane >= d)
                t = P::apply(y, t);
        }
        P wpre = t.shfl((warp + 31) & 31);
        if (warp == 0)
            wpre = P::ident();
        base[s] = P::apply(P::apply(carry, wpre), ex[s]);
        carry = P::apply(carry, t.shfl(kNW - 1));
    }

    // Warp 0: the super-tile's pair (published at once), the look-back, the
    // inclusive prefix.
    if (warp == 0) {
#if MT_RBK_EARLY
        const uint64_t aggp = sm.agg;  // published before the scan
#else
        const uint64_t aggp = ((uint64_t)carry.c << 32) | P::bits(carry.s);
        publish_aggregate<uint64_t, Op>(a.lb, g, 0, aggp);
#endif
        uint64_t pre = 0;  // the identity pair
        if (a.lb.recs != nullptr && g != 0) {
            pre = warp_lookback<uint64_t, Op, kRbkLbPerLane>(a.lb.recs, g, 0, a.lb.spin_limit);
            if (lane == 0 && g != a.lb.skip_tile)
                publish_record<uint64_t>(a.lb, g, kIncl, Op::apply(pre, aggp));
        }
        if (lane == 0)
            sm.prefix = pre;
    }
    // Does the super-tile's last element end its run?
    const bool last_ends =
        lhi > llo && (has_last || (MT_CHECK_INDEX(lhi - 1, kRbkTE) && keys_differ<KF>(knext, skey[lhi - 1])));
    const int u_last = (lhi - 1) >> 3;  // the unit of the last valid element
    __syncthreads();
    const P tp = P::unpack(sm.prefix);

    // Pass 2: heads write their key, run ends the run's sum, at run index
    // c - 1.
#pragma unroll
    for (int s = 0; s < kRbkSub; ++s) {
        const int u = s * kRbkThreads + threadIdx.x;
        const uint32_t m = mh[s];
        uint32_t e;  // element k ends a run: k + 1 starts one, or k is the last
        if (FULL) {
            const uint32_t mn = (u + 1 < kRbkUnits) ? sm.heads[u + 1] : (last_ends ? 1u : 0u);
            e = (m >> 1) | ((mn & 1u) << 7);
        } else {
            const uint32_t mn = (u + 1 < kRbkUnits) ? sm.heads[u + 1] : 0u;
            e = (m >> 1) | ((mn & 1u) << 7);
            const int li = lhi - 1 - 8 * u;
            if (li >= 0 && li < 8)
                e = (e & ((1u << li) - 1u)) | ((last_ends ? 1u : 0u) << li);
            else if (li < 0)
                e = 0u;
            const int lv = llo - 8 * u;  // elements before the first valid one end nothing
            if (lv > 0)
                e &= lv >= 8 ? 0u : ~((1u << lv) - 1u);
        }
        uint4 k0, k1, v0, v1;
        load_unit(sm.keys, u, k0, k1);
        load_unit(sm.vals, u, v0, v1);
        P run = P::apply(tp, base[s]);
        // The unit's run indices lie in [run.c - 1, run.c + popc(m) - 1]: when
        // that range is inside [0, n_live) no store needs its own check.
        const bool inside = run.c >= 1u && run.c + (uint32_t)__popc(m) <= n_live;
        auto outputs = [&](auto checked) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 8 * u + k;
                const bool h = (m >> k) & 1u;
                if (FULL || (i >= llo && i < lhi)) {
                    const V v = P::val(word8(v0, v1, k));
                    run.c += h ? 1u : 0u;
                    run.s = h ? v : run.s + v;
                }
                const uint32_t r = run.c - 1u;
                const bool ok = !decltype(checked)::value || r < n_live;
                if (h && ok && MT_CHECK_RANGE(a.keys_out + r, 4, a.keys_out, a.keys_out + n_live))
                    a.keys_out[r] = word8(k0, k1, k);
                if (((e >> k) & 1u) && ok && MT_CHECK_RANGE(a.vals_out + r, 4, a.vals_out, a.vals_out + n_live))
                    a.vals_out[r] = P::bits(run.s);
            }
        };
        if (inside)
            outputs(std::false_type{});
        else
            outputs(std::true_type{});
        if (has_last && u == u_last)
            *a.num_runs = (int32_t)(run.c <= n_live ? run.c : n_live);
    }
}

#ifndef MT_RBK_MINB
#define MT_RBK_MINB 4  // resident CTAs per SM asked of the compiler (64 registers)
#endif
template <bool KF, bool VF>
__global__ void __launch_bounds__(kRbkThreads, MT_RBK_MINB) k_reduce_by_key(RbkArgs a) {
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
    a.lb.nrec = ntiles;

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
            uint32_t bytes = (uint32_t)((cend - c0) * 16);
            if (!MT_CHECK_RANGE(&sm.keys[0], bytes, &sm.keys[0], &sm.keys[kRbkChunks]))
                bytes = 0u;  // checked build: no copies (the phase completes with no bytes)
            mbar_arrive_expect_tx(&sm.bar, 2 * bytes);
            if (bytes != 0u) {
                bulk_g2s(&sm.keys[0], vk + c0, bytes, &sm.bar);
                bulk_g2s(&sm.vals[0], vv + c0, bytes, &sm.bar);
            }
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
    a.lb.nrec = 0;  // set by the kernel
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
