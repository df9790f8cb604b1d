// mt_reduce.cu -- device-wide reduction out[0] = op(arr[0:n]) (add / min /
// max over i32, i64 and f32) with the live count read on the device.
//
// Semantics follow the Quadrants "Algorithms" user guide, section
// "qd.algorithms.reduce_{add,min,max}": the result goes to out[0], and an
// empty input gives the identity of "Semantics > Common conventions >
// Identity value". The page's realisation is a fixed-depth tree of launches;
// here one persistent kernel reads every element once: each CTA folds a
// grid-strided set of tiles into a partial, writes it to scratch, and the
// last CTA to finish (an atomic ticket) folds the partials in a fixed
// grouping, so a float sum's rounding is the same on every call.
//
// min/max keep the earliest of equal elements ((b < a) ? b : a). For integers
// equal values are identical, so any grouping gives that result. For f32 the
// two zeros compare equal but differ in sign, so f32 min/max also remember
// where their extreme came from: each thread folds its elements in index
// order with a strict comparison (a later equal element never replaces an
// earlier one) and keeps the index of the 16-byte chunk its extreme came
// from; threads and CTAs then combine 64-bit keys (the value's order in the
// high half, the chunk index in the low half, ties to the lower chunk), and
// the last CTA re-reads the winning chunk and returns its earliest element
// equal to the extreme, with that element's own bits.
#include <type_traits>

#include "mt_tile.cuh"

namespace mt {

constexpr int kRedThreads = 256;
constexpr int kRedItems = 8;  // 16-byte chunks per thread per tile: 128 bytes in flight
constexpr int kRedTileChunks = kRedThreads * kRedItems;
constexpr int kRedMaxCtas = 4096;  // partial slots in the scratch

struct RedArgs {
    const char *in;
    void *out;
    uint64_t *scratch;  // [0] ticket counter (zero at launch), then kRedMaxCtas partial slots
    const int32_t *n_dev;
};

// ---- what is folded: the value itself, or an f32 (value, index) key --------
template <class S, class Op>
struct Fold {
    using Acc = typename Codec<S>::Acc;
    using T = Acc;
    __device__ __forceinline__ static T ident() { return Op::template identity<Acc>(); }
    __device__ __forceinline__ static T make(Acc v, int64_t) { return v; }
    __device__ __forceinline__ static T apply(T a, T b) { return Op::apply(a, b); }
    __device__ __forceinline__ static uint64_t bits(T v) {
        if constexpr (sizeof(T) == 8)
            return (uint64_t)v;
        else
            return (uint64_t)bits32<T>(v);
    }
    __device__ __forceinline__ static T from(uint64_t b) {
        if constexpr (sizeof(T) == 8)
            return (T)b;
        else
            return from32<T>((uint32_t)b);
    }
};

// Order-preserving 32-bit image of an f32 in which -0 and +0 coincide.
__device__ __forceinline__ uint32_t f32_order(float v) {
    uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// f32 min/max: a float and the chunk it came from per thread; 64-bit keys
// (order, chunk) between threads. min: the smallest key wins; max: the
// largest key wins with ~chunk in the low half, so equal values still
// prefer the lower chunk.
constexpr uint32_t kNoChunk = 0xffffffffu;

struct ChunkState {
    float v;     // the thread's extreme so far
    uint32_t c;  // the chunk it came from (kNoChunk: none yet)
};

template <bool kMax>
struct ChunkFold {
    using T = uint64_t;
    using State = ChunkState;
    __device__ __forceinline__ static float ident_v() { return kMax ? -INFINITY : INFINITY; }
    __device__ __forceinline__ static bool better(float x, float v) { return kMax ? (x > v) : (x < v); }
    __device__ __forceinline__ static T ident() { return key(State{ident_v(), kNoChunk}); }
    __device__ __forceinline__ static T key(const State &st) {
        return ((uint64_t)f32_order(st.v) << 32) | (kMax ? (uint64_t)(~st.c) : (uint64_t)st.c);
    }
    __device__ __forceinline__ static uint32_t chunk(T k) { return kMax ? ~(uint32_t)k : (uint32_t)k; }
    __device__ __forceinline__ static uint32_t order(T k) { return (uint32_t)(k >> 32); }
    __device__ __forceinline__ static T apply(T a, T b) { return kMax ? (b > a ? b : a) : (b < a ? b : a); }
    __device__ __forceinline__ static uint64_t bits(T v) { return v; }
    __device__ __forceinline__ static T from(uint64_t b) { return b; }
};

template <class S, class Op>
struct FoldOf {
    using type = Fold<S, Op>;
};
template <>
struct FoldOf<float, OpMin> {
    using type = ChunkFold<false>;
};
template <>
struct FoldOf<float, OpMax> {
    using type = ChunkFold<true>;
};
template <class F>
constexpr bool kChunkFold = std::is_same<F, ChunkFold<false>>::value || std::is_same<F, ChunkFold<true>>::value;

template <class F>
__device__ __forceinline__ typename F::T block_fold(typename F::T v, typename F::T *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        v = F::apply(v, __shfl_down_sync(kFull, v, d));  // lane order kept: lower lanes left
    if (lane == 0)
        sm[warp] = v;
    __syncthreads();
    typename F::T r = F::ident();
#pragma unroll
    for (int w = 0; w < kRedThreads / 32; ++w)
        r = F::apply(r, sm[w]);
    __syncthreads();
    return r;
}

template <class S, class Op>
__global__ void __launch_bounds__(kRedThreads, sizeof(S) == 8 ? 2 : 4) k_reduce(RedArgs a) {
    pdl_prologue();
    using C = Codec<S>;
    using Acc = typename C::Acc;
    using F = typename FoldOf<S, Op>::type;
    using T = typename F::T;
    constexpr int E = C::E;
    constexpr int64_t s = sizeof(S);
    __shared__ T sm[kRedThreads / 32];
    __shared__ bool last;

    const int32_t n32 = *a.n_dev;
    const int64_t n = n32 > 0 ? n32 : 0;
    const int64_t head = (int64_t)(((uintptr_t)a.in & 15u) / s);
    const uint4 *vin = reinterpret_cast<const uint4 *>(a.in - head * s);
    const int64_t lo = head, hi = head + n;
    const int64_t nchunks = n > 0 ? (hi + E - 1) / E : 0;  // no element: touch nothing

    T acc = F::ident();
    [[maybe_unused]] ChunkState st{0.0f, kNoChunk};
    if constexpr (kChunkFold<F>)
        st.v = F::ident_v();
    for (int64_t t = blockIdx.x; t * kRedTileChunks < nchunks; t += gridDim.x) {
        const int64_t c0 = t * kRedTileChunks;
        const bool full = c0 * E >= lo && (c0 + kRedTileChunks) * E <= hi;
        uint4 raw[kRedItems];
#pragma unroll
        for (int j = 0; j < kRedItems; ++j) {
            const int64_t c = c0 + j * kRedThreads + threadIdx.x;
            raw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (full || c < nchunks)
                raw[j] = ld_stream(vin + c);
        }
#pragma unroll
        for (int j = 0; j < kRedItems; ++j) {
            const int64_t c = c0 + j * kRedThreads + threadIdx.x;
            const int64_t v0 = c * E;
            Acc x[E];
            C::unpack(raw[j], x);
            if constexpr (kChunkFold<F>) {
                // the chunk's extreme, earliest first; then the thread's
                float m = F::ident_v();
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if ((full || (v0 + k >= lo && v0 + k < hi)) && F::better(x[k], m))
                        m = x[k];
                if (F::better(m, st.v)) {
                    st.v = m;
                    st.c = (uint32_t)c;
                }
            } else {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (full || (v0 + k >= lo && v0 + k < hi))
                        acc = F::apply(acc, F::make(x[k], v0 + k - head));
            }
        }
    }
    if constexpr (kChunkFold<F>)
        acc = F::key(st);
    const T part = block_fold<F>(acc, sm);

    // Partial to scratch; the last CTA to arrive folds all partials in order.
    if (threadIdx.x == 0) {
        st_relaxed_u64(a.scratch + kHeaderSlots + blockIdx.x, F::bits(part));
        __threadfence();
        const unsigned long long ticket = atomicAdd(reinterpret_cast<unsigned long long *>(a.scratch), 1ull);
        last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!last)
        return;
    __threadfence();
    T r = F::ident();
    // thread i folds partials i, i + 256, ...; the block fold then combines the
    // threads in a fixed tree: the same grouping on every call.
    for (int i = threadIdx.x; i < (int)gridDim.x; i += kRedThreads)
        r = F::apply(r, F::from(ld_relaxed_u64(a.scratch + kHeaderSlots + i)));
    r = block_fold<F>(r, sm);
    if (threadIdx.x == 0) {
        if constexpr (!kChunkFold<F>) {
            *static_cast<S *>(a.out) = (S)r;
        } else {
            // the earliest element of the winning chunk equal to the extreme,
            // with its own bits; no such chunk: the identity (or an infinity
            // equal to it)
            float res = F::ident_v();
            const uint32_t c = F::chunk(r);
            if (c != kNoChunk) {
                Acc x[E];
                C::unpack(ld_stream(vin + c), x);
                bool found = false;
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const int64_t v = (int64_t)c * E + k;
                    if (!found && v >= lo && v < hi && f32_order(x[k]) == F::order(r)) {
                        res = x[k];
                        found = true;
                    }
                }
            }
            *static_cast<float *>(a.out) = res;
        }
        a.scratch[0] = 0ull;  // the ticket counter, ready for the next call
    }
}

template <class S, class Op>
static cudaError_t launch_reduce(const RedArgs &a, const Launch &L) {
    static int per_sm[128] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 128)
        return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_reduce<S, Op>, kRedThreads, 0);
        if (e != cudaSuccess)
            return e;
        per_sm[dev] = b > 0 ? b : 1;
    }
    int64_t grid = (int64_t)L.sm_count * per_sm[dev];
    if (grid > kRedMaxCtas)
        grid = kRedMaxCtas;
    e = launch_pdl(k_reduce<S, Op>, (unsigned)grid, kRedThreads, 0, L.stream, a);
    note_launch();
    return e;
}

int64_t reduce_scratch_slots() { return kHeaderSlots + kRedMaxCtas; }

template <class S>
static cudaError_t reduce_op(int op, const RedArgs &a, const Launch &L) {
    switch (op) {
    case 0: return launch_reduce<S, OpAdd>(a, L);
    case 1: return launch_reduce<S, OpMin>(a, L);
    case 2: return launch_reduce<S, OpMax>(a, L);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t reduce_launch(const void *arr, void *out, uint64_t *scratch, const int32_t *n_dev,
                          int dtype, int op, const Launch &L) {
    RedArgs a;
    a.in = static_cast<const char *>(arr);
    a.out = out;
    a.scratch = scratch;
    a.n_dev = n_dev;
    switch (dtype) {
    case 0: return reduce_op<float>(op, a, L);
    case 3: return reduce_op<int32_t>(op, a, L);
    case 4: return reduce_op<int64_t>(op, a, L);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mt
