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
// open run). Tiles are chained by the decoupled look-back on that pair
// (packed in 64 bits), so every run's sum is complete at its last element:
// heads write keys_out[c - 1], run ends write values_out[c - 1]. No atomics
// on the outputs, and sums are added in a fixed order.
#include "mt_lookback.cuh"

namespace mt {

constexpr int kRbkThreads = 256;
constexpr int kRbkItems = 4;                                       // 16-byte chunks per thread
constexpr int kRbkChunks = kRbkThreads * kRbkItems;                // per tile
constexpr int64_t kRbkTE = (int64_t)kRbkChunks * 4;                // elements per tile (4096)

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

template <bool KF>
__device__ __forceinline__ bool keys_differ(uint32_t a, uint32_t b) {
    if (KF)
        return __uint_as_float(a) != __uint_as_float(b);  // NaN differs from everything
    return a != b;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

template <bool KF, bool VF>
__global__ void __launch_bounds__(kRbkThreads) k_reduce_by_key(RbkArgs a) {
    pdl_prologue();
    using Op = SegOp<VF>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int kNW = kRbkThreads / 32;
    __shared__ uint64_t warp_tot[2][kNW];
    __shared__ uint64_t prefix[2];
    __shared__ unsigned long long tile_id;

    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t head = (int64_t)(((uintptr_t)a.keys & 15u) / 4);
    const uint4 *vk = reinterpret_cast<const uint4 *>(a.keys - head * 4);
    const uint4 *vv = reinterpret_cast<const uint4 *>(a.vals - head * 4);
    const uint32_t *ek = reinterpret_cast<const uint32_t *>(a.keys) - head;  // virtual element 0
    const int64_t lo = head, hi = head + n;
    const int64_t ntiles = n > 0 ? (hi + kRbkTE - 1) / kRbkTE : 0;

    for (int64_t it = 0;; ++it) {
        if (threadIdx.x == 0)
            tile_id = atomicAdd(a.counter, 1ull);
        __syncthreads();  // tile id visible; every thread is done with the last tile's shared state
        const int64_t g = (int64_t)tile_id;
        if (g >= ntiles)
            break;
        const int buf = (int)(it & 1);
        const int64_t t0 = g * kRbkTE;

        // Loads: keys and values of this thread's chunks, and for each chunk
        // the key before it and the key after it (neighbours' chunks: L1/L2).
        uint4 kr[kRbkItems], vr[kRbkItems];
        uint32_t kprev[kRbkItems], knext[kRbkItems];
#pragma unroll
        for (int j = 0; j < kRbkItems; ++j) {
            const int c = warp * 32 * kRbkItems + j * 32 + lane;
            const int64_t v0 = t0 + (int64_t)c * 4;
            kr[j] = vr[j] = make_uint4(0u, 0u, 0u, 0u);
            kprev[j] = knext[j] = 0u;
            if (v0 < hi && v0 + 4 > lo) {
                kr[j] = ld_stream(vk + v0 / 4);
                vr[j] = ld_stream(vv + v0 / 4);
            }
            if (v0 - 1 >= lo && v0 - 1 < hi)
                kprev[j] = __ldg(ek + v0 - 1);
            if (v0 + 4 >= lo && v0 + 4 < hi)
                knext[j] = __ldg(ek + v0 + 4);
        }

        // Per element: the pair (head, value); serial inclusive scan per chunk.
        uint64_t x[kRbkItems][4];
        bool endf[kRbkItems][4], headf[kRbkItems][4];
#pragma unroll
        for (int j = 0; j < kRbkItems; ++j) {
            const int c = warp * 32 * kRbkItems + j * 32 + lane;
            const int64_t v0 = t0 + (int64_t)c * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t v = v0 + k;
                const bool valid = v >= lo && v < hi;
                const uint32_t key = word(kr[j], k);
                const uint32_t before = k == 0 ? kprev[j] : word(kr[j], k - 1);
                const uint32_t after = k == 3 ? knext[j] : word(kr[j], k + 1);
                const bool h = valid && (v == lo || keys_differ<KF>(key, before));
                headf[j][k] = h;
                endf[j][k] = valid && (v == hi - 1 || keys_differ<KF>(after, key));
                // invalid elements are the identity (0, 0)
                x[j][k] = valid ? (((uint64_t)(h ? 1u : 0u) << 32) | word(vr[j], k)) : 0ull;
            }
#pragma unroll
            for (int k = 1; k < 4; ++k)
                x[j][k] = Op::apply(x[j][k - 1], x[j][k]);
        }

        // Warp scans of the chunk totals (one per j), then the run over j.
        uint64_t inc[kRbkItems];
#pragma unroll
        for (int j = 0; j < kRbkItems; ++j)
            inc[j] = x[j][3];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
            for (int j = 0; j < kRbkItems; ++j) {
                const uint64_t y = __shfl_up_sync(kFull, inc[j], d);
                if (lane >= d)
                    inc[j] = Op::apply(y, inc[j]);
            }
        }
        uint64_t pre[kRbkItems];
        uint64_t run = 0ull;
#pragma unroll
        for (int j = 0; j < kRbkItems; ++j) {
            uint64_t e = __shfl_up_sync(kFull, inc[j], 1);
            if (lane == 0)
                e = 0ull;
            pre[j] = Op::apply(run, e);
            run = Op::apply(run, __shfl_sync(kFull, inc[j], 31));
        }
        if (lane == 0)
            warp_tot[buf][warp] = run;
        __syncthreads();
        uint64_t wpre = 0ull, agg = 0ull;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            const uint64_t t = warp_tot[buf][w];
            if (w < warp)
                wpre = Op::apply(wpre, t);
            agg = Op::apply(agg, t);
        }

        // The tile's prefix: (runs started before it, sum of the run open at
        // its start); the first tile's is the identity.
        const uint64_t tp = tile_prefix<uint64_t, Op>(a.lb, g, 0, agg, &prefix[buf]);
        const uint64_t base0 = Op::apply(tp, wpre);

        // Heads write their key, run ends the run's sum, at run index c - 1.
#pragma unroll
        for (int j = 0; j < kRbkItems; ++j) {
            const uint64_t base = Op::apply(base0, pre[j]);
            const int c = warp * 32 * kRbkItems + j * 32 + lane;
            const int64_t v0 = t0 + (int64_t)c * 4;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t p = Op::apply(base, x[j][k]);
                const uint32_t r = (uint32_t)(p >> 32) - 1u;
                if (headf[j][k])
                    a.keys_out[r] = word(kr[j], k);
                if (endf[j][k]) {
                    a.vals_out[r] = (uint32_t)p;
                    if (v0 + k == hi - 1)
                        *a.num_runs = (int32_t)(r + 1u);
                }
            }
        }
    }
}

template <bool KF, bool VF>
static cudaError_t launch_rbk(const RbkArgs &a, const Launch &L) {
    static int per_sm[128] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_reduce_by_key<KF, VF>, kRbkThreads, 0);
        if (e != cudaSuccess)
            return e;
        per_sm[dev] = b > 0 ? b : 1;
    }
    e = launch_pdl(k_reduce_by_key<KF, VF>, (unsigned)(L.sm_count * per_sm[dev]), kRbkThreads, 0, L.stream, a);
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
