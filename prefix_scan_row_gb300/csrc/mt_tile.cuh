// mt_tile.cuh -- device building blocks shared by the scan kernels (sm_103a).
//
// One CTA tile is 256 threads x ITEMS chunks of 16 bytes. A warp owns a
// contiguous run of 32*ITEMS chunks and reads it "warp-striped": chunk j of
// lane l is chunk 32*j + l of the warp's run, so each 16-byte vector load or
// store instruction of a warp touches 512 contiguous bytes.
//
// Scan hierarchy inside a tile (all combines keep the element order, the
// "ordered tree" of LuisaCompute "Tile operations and reductions", section
// "Why not just infer it from reduce?"):
//   1. each thread scans the E elements of each of its chunks in registers;
//   2. for each j, an inclusive warp scan (shfl_up) of the chunk totals;
//   3. a running carry across j inside the warp;
//   4. warp totals through shared memory to a block-wide exclusive prefix;
//   5. a single-pass decoupled look-back across tiles of the same segment
//      (row or 1-D array) gives the tile's exclusive prefix; the Quadrants
//      "Algorithms" guide, section "Related", names decoupled look-back as
//      the more efficient alternative to a multi-pass scan.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mt_internal.h"

namespace mt {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

// Look-back status flags of a tile record.
constexpr uint32_t kEmpty = 0;  // nothing published yet (the reset state)
constexpr uint32_t kAgg = 1;    // the tile's own aggregate is published
constexpr uint32_t kIncl = 2;   // the inclusive prefix through this tile is published

constexpr int kErrTimeout = -5;  // same value as MT_ERR_LOOKBACK_TIMEOUT
constexpr uint32_t kCopyWaitLimit = 1u << 26;  // mbarrier polls before a copy is given up

// Per translation unit device error word; written when a look-back wait gives up.
static __device__ int g_mt_err;

// ---------------------------------------------------------------------------
// Bounds-checked build. Compiled with MT_CHECKED=1, every global store and
// every shared-memory access of the kernels is first checked against the
// buffer it belongs to; an access outside it records MT_ERR_BOUNDS in the
// device error word and is skipped (a load then yields zero). Nothing traps,
// so a bad index shows up in mt_scan_status() and the context stays usable.
// In the ordinary build the checks are the constant `true` and cost nothing.
// ---------------------------------------------------------------------------
#ifndef MT_CHECKED
#define MT_CHECKED 0
#endif
constexpr int kErrBounds = -9;  // same value as MT_ERR_BOUNDS

__device__ __forceinline__ bool check_index(long long i, long long n) {
    if (i >= 0 && i < n)
        return true;
    atomicCAS(&g_mt_err, 0, kErrBounds);
    return false;
}
// [p, p + bytes) inside [lo, hi)
__device__ __forceinline__ bool check_range(const void *p, unsigned long long bytes, const void *lo, const void *hi) {
    const uintptr_t a = (uintptr_t)p, l = (uintptr_t)lo, h = (uintptr_t)hi;
    if (a >= l && a <= h && bytes <= (unsigned long long)(h - a))
        return true;
    atomicCAS(&g_mt_err, 0, kErrBounds);
    return false;
}
#if MT_CHECKED
#define MT_CHECK_INDEX(i, n) ::mt::check_index((long long)(i), (long long)(n))
#define MT_CHECK_RANGE(p, bytes, lo, hi) ::mt::check_range((p), (bytes), (lo), (hi))
#else
#define MT_CHECK_INDEX(i, n) true
#define MT_CHECK_RANGE(p, bytes, lo, hi) true
#endif

// ---------------------------------------------------------------------------
// Combine operators. apply(a, b): `a` covers earlier elements than `b`.
// ---------------------------------------------------------------------------
template <class T> struct Lim;
template <> struct Lim<float> {
    __device__ __forceinline__ static float hi() { return __int_as_float(0x7f800000); }   // +inf
    __device__ __forceinline__ static float lo() { return __int_as_float((int)0xff800000u); }  // -inf
};
template <> struct Lim<double> {
    __device__ __forceinline__ static double hi() { return __longlong_as_double(0x7ff0000000000000ll); }  // +inf
    __device__ __forceinline__ static double lo() { return __longlong_as_double((long long)0xfff0000000000000ull); }
};
template <> struct Lim<uint32_t> {
    __device__ __forceinline__ static uint32_t hi() { return 0xffffffffu; }
    __device__ __forceinline__ static uint32_t lo() { return 0u; }
};
template <> struct Lim<uint64_t> {
    __device__ __forceinline__ static uint64_t hi() { return 0xffffffffffffffffull; }
    __device__ __forceinline__ static uint64_t lo() { return 0ull; }
};
template <> struct Lim<int32_t> {
    __device__ __forceinline__ static int32_t hi() { return 0x7fffffff; }
    __device__ __forceinline__ static int32_t lo() { return (int32_t)0x80000000u; }
};
template <> struct Lim<int64_t> {
    __device__ __forceinline__ static int64_t hi() { return 0x7fffffffffffffffll; }
    __device__ __forceinline__ static int64_t lo() { return (int64_t)0x8000000000000000ull; }
};

struct OpAdd {
    template <class T> __device__ __forceinline__ static T identity() { return T(0); }
    __device__ __forceinline__ static float apply(float a, float b) { return a + b; }
    __device__ __forceinline__ static uint32_t apply(uint32_t a, uint32_t b) { return a + b; }
    // integer add wraps modulo 2^width (two's complement), done in unsigned arithmetic
    __device__ __forceinline__ static int32_t apply(int32_t a, int32_t b) {
        return (int32_t)((uint32_t)a + (uint32_t)b);
    }
    __device__ __forceinline__ static int64_t apply(int64_t a, int64_t b) {
        return (int64_t)((uint64_t)a + (uint64_t)b);
    }
    __device__ __forceinline__ static uint64_t apply(uint64_t a, uint64_t b) { return a + b; }
    __device__ __forceinline__ static double apply(double a, double b) { return a + b; }
};

// min/max keep the earlier operand on ties, so any grouping gives the same
// bits as a left-to-right fold (the leftmost extreme element).
struct OpMin {
    template <class T> __device__ __forceinline__ static T identity() { return Lim<T>::hi(); }
    template <class T> __device__ __forceinline__ static T apply(T a, T b) { return (b < a) ? b : a; }
};
struct OpMax {
    template <class T> __device__ __forceinline__ static T identity() { return Lim<T>::lo(); }
    template <class T> __device__ __forceinline__ static T apply(T a, T b) { return (b > a) ? b : a; }
};
// Product (the row scans' prod variant; f32 accumulation only).
struct OpMul {
    template <class T> __device__ __forceinline__ static T identity() { return T(1); }
    __device__ __forceinline__ static float apply(float a, float b) { return a * b; }
};

// ---------------------------------------------------------------------------
// Storage codecs: a 16-byte chunk <-> E accumulator values.
// bf16/f16 widen exactly to f32 and narrow with round-to-nearest-even
// (LuisaCompute "Tile operations and reductions", "Storage and arithmetic
// precision"); the metaltile-std scan.rs kernels likewise load as f32 and
// cast once at the store.
// ---------------------------------------------------------------------------
template <class S> struct Codec;

template <> struct Codec<float> {
    using Acc = float;
    static constexpr int E = 4;
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                          __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
    __device__ __forceinline__ static Acc load1(const float *p) { return *p; }
    __device__ __forceinline__ static void store1(float *p, Acc v) { *p = v; }
};

template <> struct Codec<__nv_bfloat16> {
    using Acc = float;
    static constexpr int E = 8;
    __device__ __forceinline__ static void two(uint32_t w, Acc &a, Acc &b) {
        a = __uint_as_float(w << 16);          // bf16 is the top half of an f32
        b = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack2(Acc a, Acc b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half)
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        two(v.x, x[0], x[1]); two(v.y, x[2], x[3]); two(v.z, x[4], x[5]); two(v.w, x[6], x[7]);
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
    }
    __device__ __forceinline__ static Acc load1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ __forceinline__ static void store1(__nv_bfloat16 *p, Acc v) { *p = __float2bfloat16_rn(v); }
};

template <> struct Codec<__half> {
    using Acc = float;
    static constexpr int E = 8;
    __device__ __forceinline__ static void two(uint32_t w, Acc &a, Acc &b) {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        float2 f = __half22float2(h);
        a = f.x; b = f.y;
    }
    __device__ __forceinline__ static uint32_t pack2(Acc a, Acc b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        two(v.x, x[0], x[1]); two(v.y, x[2], x[3]); two(v.z, x[4], x[5]); two(v.w, x[6], x[7]);
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
    }
    __device__ __forceinline__ static Acc load1(const __half *p) { return __half2float(*p); }
    __device__ __forceinline__ static void store1(__half *p, Acc v) { *p = __float2half_rn(v); }
};

template <> struct Codec<int32_t> {
    using Acc = int32_t;
    static constexpr int E = 4;
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        x[0] = (int32_t)v.x; x[1] = (int32_t)v.y; x[2] = (int32_t)v.z; x[3] = (int32_t)v.w;
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4((uint32_t)x[0], (uint32_t)x[1], (uint32_t)x[2], (uint32_t)x[3]);
    }
    __device__ __forceinline__ static Acc load1(const int32_t *p) { return *p; }
    __device__ __forceinline__ static void store1(int32_t *p, Acc v) { *p = v; }
};

template <> struct Codec<int64_t> {
    using Acc = int64_t;
    static constexpr int E = 2;
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        x[0] = (int64_t)(((uint64_t)v.y << 32) | v.x);
        x[1] = (int64_t)(((uint64_t)v.w << 32) | v.z);
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4((uint32_t)x[0], (uint32_t)((uint64_t)x[0] >> 32),
                          (uint32_t)x[1], (uint32_t)((uint64_t)x[1] >> 32));
    }
    __device__ __forceinline__ static Acc load1(const int64_t *p) { return *p; }
    __device__ __forceinline__ static void store1(int64_t *p, Acc v) { *p = v; }
};

template <> struct Codec<uint32_t> {
    using Acc = uint32_t;
    static constexpr int E = 4;
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) { return make_uint4(x[0], x[1], x[2], x[3]); }
    __device__ __forceinline__ static Acc load1(const uint32_t *p) { return *p; }
    __device__ __forceinline__ static void store1(uint32_t *p, Acc v) { *p = v; }
};

template <> struct Codec<uint64_t> {
    using Acc = uint64_t;
    static constexpr int E = 2;
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        x[0] = ((uint64_t)v.y << 32) | v.x;
        x[1] = ((uint64_t)v.w << 32) | v.z;
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4((uint32_t)x[0], (uint32_t)(x[0] >> 32), (uint32_t)x[1], (uint32_t)(x[1] >> 32));
    }
    __device__ __forceinline__ static Acc load1(const uint64_t *p) { return *p; }
    __device__ __forceinline__ static void store1(uint64_t *p, Acc v) { *p = v; }
};

template <> struct Codec<double> {
    using Acc = double;
    static constexpr int E = 2;
    __device__ __forceinline__ static void unpack(const uint4 &v, Acc (&x)[E]) {
        x[0] = __hiloint2double((int)v.y, (int)v.x);
        x[1] = __hiloint2double((int)v.w, (int)v.z);
    }
    __device__ __forceinline__ static uint4 pack(const Acc (&x)[E]) {
        return make_uint4((uint32_t)__double2loint(x[0]), (uint32_t)__double2hiint(x[0]),
                          (uint32_t)__double2loint(x[1]), (uint32_t)__double2hiint(x[1]));
    }
    __device__ __forceinline__ static Acc load1(const double *p) { return *p; }
    __device__ __forceinline__ static void store1(double *p, Acc v) { *p = v; }
};

// ---------------------------------------------------------------------------
// Memory primitives (inline PTX).
// ---------------------------------------------------------------------------
// Streaming 16-byte load that does not allocate in L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_v4(uint4 *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_i32(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---- shared-memory barriers and bulk (TMA) copies ----------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
// One 16-byte shared-memory access as a single instruction: a 16-byte chunk
// read as two 8-byte halves costs a warp twice the wavefronts.
__device__ __forceinline__ uint4 lds128(const uint4 *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(p)) : "memory");
    return v;
}
__device__ __forceinline__ void sts128(uint4 *p, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "r"(smem_addr(p)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}
// Makes barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before
// later bulk-copy writes into the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// Asynchronous 4- or 8-byte copy global -> shared: no register holds the
// value while it is in flight, so a thread can have many outstanding.
// Both addresses aligned to the size; complete after cp_async_wait_all().
template <int BYTES>
__device__ __forceinline__ void cp_async_small(void *dst, const void *src) {
    static_assert(BYTES == 4 || BYTES == 8, "4- or 8-byte copies");
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" :: "r"(smem_addr(dst)), "l"(src), "n"(BYTES)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Bounded wait for phase `parity` of `bar`; false if it did not complete.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

template <class T> __device__ __forceinline__ uint32_t bits32(T v);
template <> __device__ __forceinline__ uint32_t bits32<float>(float v) { return __float_as_uint(v); }
template <> __device__ __forceinline__ uint32_t bits32<int32_t>(int32_t v) { return (uint32_t)v; }
template <> __device__ __forceinline__ uint32_t bits32<uint32_t>(uint32_t v) { return v; }
template <class T> __device__ __forceinline__ T from32(uint32_t b);
template <> __device__ __forceinline__ float from32<float>(uint32_t b) { return __uint_as_float(b); }
template <> __device__ __forceinline__ int32_t from32<int32_t>(uint32_t b) { return (int32_t)b; }
template <> __device__ __forceinline__ uint32_t from32<uint32_t>(uint32_t b) { return b; }
// 8-byte values as raw bits (status records, partials).
template <class T> __device__ __forceinline__ uint64_t bits64(T v);
template <> __device__ __forceinline__ uint64_t bits64<int64_t>(int64_t v) { return (uint64_t)v; }
template <> __device__ __forceinline__ uint64_t bits64<uint64_t>(uint64_t v) { return v; }
template <> __device__ __forceinline__ uint64_t bits64<double>(double v) { return (uint64_t)__double_as_longlong(v); }
template <class T> __device__ __forceinline__ T from64(uint64_t b);
template <> __device__ __forceinline__ int64_t from64<int64_t>(uint64_t b) { return (int64_t)b; }
template <> __device__ __forceinline__ uint64_t from64<uint64_t>(uint64_t b) { return b; }
template <> __device__ __forceinline__ double from64<double>(uint64_t b) { return __longlong_as_double((long long)b); }

}  // namespace mt
