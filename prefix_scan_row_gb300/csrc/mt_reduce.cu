// mt_reduce.cu -- device-wide reduction out[0] = op(arr[0:n]) (add / min /
// max over i32, i64, u32, u64, f32 and f64) with the live count read on the
// device.
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
// equal values are identical, so any grouping gives that result. For floats
// the two zeros compare equal but differ in sign, so f32/f64 min/max also
// remember where their extreme came from: each thread folds its elements in
// index order with a strict comparison (a later equal element never replaces
// an earlier one) and keeps the index of the 16-byte chunk its extreme came
// from; threads and CTAs then combine (order, chunk) pairs -- the value's
// order-preserving image, ties to the lower chunk -- and the last CTA
// re-reads the winning chunk and returns its earliest element equal to the
// extreme, with that element's own bits.
#include <type_traits>

#include "mt_tile.cuh"

namespace mt {

constexpr int kRedThreads = 256;
constexpr int kRedItems = 8;  // 16-byte chunks per thread per tile: 128 bytes in flight
constexpr int kRedTileChunks = kRedThreads * kRedItems;
constexpr int kRedMaxCtas = 4096;   // partials in the scratch
constexpr int kRedPartialSlots = 2;  // 8-byte slots per partial (a pair needs two)
#ifndef MT_RED_F64_ACCS
#define MT_RED_F64_ACCS 8
#endif
// Independent running sums per thread for f64 adds: GB300's FP64 adds are
// few and slow, and one chain per thread leaves the pipe waiting on results.
constexpr int kRedF64Accs = MT_RED_F64_ACCS;

struct RedArgs {
    const char *in;
    void *out;
    uint64_t *scratch;  // [0] ticket counter (zero at launch), then kRedMaxCtas partials
    const int32_t *n_dev;
};

// ---- what is folded -----------------------------------------------------------
// The value itself (integers; float sums).
template <class S, class Op>
struct Fold {
    using Acc = typename Codec<S>::Acc;
    using T = Acc;
    __device__ __forceinline__ static T ident() { return Op::template identity<Acc>(); }
    __device__ __forceinline__ static T apply(T a, T b) { return Op::apply(a, b); }
    __device__ __forceinline__ static T shfl_down(T v, int d) { return __shfl_down_sync(kFull, v, d); }
    __device__ __forceinline__ static void store(uint64_t *p, T v) {
        if constexpr (sizeof(T) == 8)
            st_relaxed_u64(p, bits64<T>(v));
        else
            st_relaxed_u64(p, (uint64_t)bits32<T>(v));
    }
    __device__ __forceinline__ static T load(const uint64_t *p) {
        if constexpr (sizeof(T) == 8)
            return from64<T>(ld_relaxed_u64(p));
        else
            return from32<T>((uint32_t)ld_relaxed_u64(p));
    }
};

// Order-preserving unsigned images of f32 / f64 in which -0 and +0 coincide.
__device__ __forceinline__ uint64_t float_order(float v) {
    const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t float_order(double v) {
    const uint64_t u = (uint64_t)__double_as_longlong(v == 0.0 ? 0.0 : v);
    return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

constexpr uint32_t kNoChunk = 0xffffffffu;

// A float's extreme and the chunk it came from (kNoChunk: none yet).
template <class V>
struct ChunkState {
    V v;
    uint32_t c;
};

// f32/f64 min/max: threads fold ChunkState; between threads and CTAs an
// (order, chunk) pair, the better order winning and equal orders going to
// the lower chunk.
template <class V, bool kMax>
struct ChunkFold {
    struct T {
        uint64_t o;  // float_order of the extreme
        uint32_t c;  // its chunk
    };
    __device__ __forceinline__ static V ident_v() { return kMax ? Lim<V>::lo() : Lim<V>::hi(); }
    __device__ __forceinline__ static bool better(V x, V v) { return kMax ? (x > v) : (x < v); }
    __device__ __forceinline__ static T pair(const ChunkState<V> &st) { return T{float_order(st.v), st.c}; }
    __device__ __forceinline__ static T ident() { return T{float_order(ident_v()), kNoChunk}; }
    __device__ __forceinline__ static T apply(T a, T b) {
        const bool take_b = (kMax ? (b.o > a.o) : (b.o < a.o)) || (b.o == a.o && b.c < a.c);
        return take_b ? b : a;
    }
    __device__ __forceinline__ static T shfl_down(T v, int d) {
        return T{__shfl_down_sync(kFull, v.o, d), __shfl_down_sync(kFull, v.c, d)};
    }
    __device__ __forceinline__ static void store(uint64_t *p, T v) {
        st_relaxed_u64(p, v.o);
        st_relaxed_u64(p + 1, (uint64_t)v.c);
    }
    __device__ __forceinline__ static T load(const uint64_t *p) {
        return T{ld_relaxed_u64(p), (uint32_t)ld_relaxed_u64(p + 1)};
    }
};

template <class S, class Op>
struct FoldOf {
    using type = Fold<S, Op>;
};
template <> struct FoldOf<float, OpMin> { using type = ChunkFold<float, false>; };
template <> struct FoldOf<float, OpMax> { using type = ChunkFold<float, true>; };
template <> struct FoldOf<double, OpMin> { using type = ChunkFold<double, false>; };
template <> struct FoldOf<double, OpMax> { using type = ChunkFold<double, true>; };

template <class F>
struct IsChunkFold : std::false_type {};
template <class V, bool kMax>
struct IsChunkFold<ChunkFold<V, kMax>> : std::true_type {};

template <class F>
__device__ __forceinline__ typename F::T block_fold(typename F::T v, typename F::T *sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        v = F::apply(v, F::shfl_down(v, d));  // lower lanes stay the left operand
    if (lane == 0 && MT_CHECK_INDEX(warp, kRedThreads / 32))
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
    constexpr bool kChunk = IsChunkFold<F>::value;
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

    constexpr int kAccs = (!kChunk && std::is_same<Acc, double>::value) ? kRedF64Accs : 1;
    T accs[kAccs];
#pragma unroll
    for (int i = 0; i < kAccs; ++i)
        accs[i] = F::ident();
    [[maybe_unused]] ChunkState<Acc> st{Acc(0), kNoChunk};
    if constexpr (kChunk)
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
            if constexpr (kChunk) {
                // each element against the thread's extreme (one compare per
                // element: GB300 compares f64 on its narrow FP64 pipe); strict,
                // so the earliest chunk with the extreme is kept
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if ((full || (v0 + k >= lo && v0 + k < hi)) && F::better(x[k], st.v)) {
                        st.v = x[k];
                        st.c = (uint32_t)c;
                    }
            } else {
#pragma unroll
                for (int k = 0; k < E; ++k)
                    if (full || (v0 + k >= lo && v0 + k < hi))
                        accs[(j * E + k) % kAccs] = F::apply(accs[(j * E + k) % kAccs], x[k]);
            }
        }
    }
    T acc = accs[0];
#pragma unroll
    for (int i = 1; i < kAccs; ++i)
        acc = F::apply(acc, accs[i]);
    if constexpr (kChunk)
        acc = F::pair(st);
    const T part = block_fold<F>(acc, sm);

    // Partial to scratch; the last CTA to arrive folds all partials.
    if (threadIdx.x == 0) {
        if (MT_CHECK_INDEX(blockIdx.x, kRedMaxCtas))
            F::store(a.scratch + kHeaderSlots + kRedPartialSlots * blockIdx.x, part);
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
        if (MT_CHECK_INDEX(i, kRedMaxCtas))
            r = F::apply(r, F::load(a.scratch + kHeaderSlots + kRedPartialSlots * i));
    r = block_fold<F>(r, sm);
    if (threadIdx.x == 0) {
        if constexpr (!kChunk) {
            *static_cast<S *>(a.out) = (S)r;
        } else {
            // the earliest element of the winning chunk equal to the extreme,
            // with its own bits; no such chunk: the identity (or an infinity
            // equal to it)
            Acc res = F::ident_v();
            if (r.c != kNoChunk) {
                Acc x[E];
                C::unpack(ld_stream(vin + r.c), x);
                bool found = false;
#pragma unroll
                for (int k = 0; k < E; ++k) {
                    const int64_t v = (int64_t)r.c * E + k;
                    if (!found && v >= lo && v < hi && float_order(x[k]) == r.o) {
                        res = x[k];
                        found = true;
                    }
                }
            }
            *static_cast<S *>(a.out) = res;
        }
        a.scratch[0] = 0ull;  // the ticket counter, ready for the next call
    }
}

template <class S, class Op>
static cudaError_t launch_reduce(const RedArgs &a, const Launch &L) {
    static PerDevice per_sm;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    int blocks = per_sm.get(dev);
    if (blocks == 0) {
        int b = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_reduce<S, Op>, kRedThreads, 0);
        if (e != cudaSuccess)
            return e;
        blocks = b > 0 ? b : 1;
        per_sm.set(dev, blocks);
    }
    int64_t grid = (int64_t)L.sm_count * blocks;
    if (grid > kRedMaxCtas)
        grid = kRedMaxCtas;
    e = launch_pdl(k_reduce<S, Op>, (unsigned)grid, kRedThreads, 0, L.stream, a);
    note_launch();
    return e;
}

int64_t reduce_scratch_slots() { return kHeaderSlots + (int64_t)kRedPartialSlots * kRedMaxCtas; }

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
    case 5: return reduce_op<uint32_t>(op, a, L);
    case 6: return reduce_op<uint64_t>(op, a, L);
    case 7: return reduce_op<double>(op, a, L);
    default: return cudaErrorInvalidValue;
    }
}

// Reads and clears this translation unit's device error word (set only by
// the bounds-checked build's checks).
cudaError_t reduce_take_error(int *code) {
    const int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mt_err, sizeof(int));
    if (e != cudaSuccess)
        return e;
    return cudaMemcpyToSymbol(g_mt_err, &zero, sizeof(int));
}

}  // namespace mt
