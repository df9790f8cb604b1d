/*
 * mt_scan.h -- C ABI of libmtscan.so, a prefix-scan library for one NVIDIA
 * GB300 GPU (sm_103a).
 *
 * All calls take plain pointers and sizes. Device pointers are CUDA device
 * (or managed) memory owned by the caller. `stream` is a cudaStream_t passed
 * as `void*`; NULL means the legacy default stream. Every call only enqueues
 * work on `stream` and returns without synchronising, except
 * mt_scan_status(), which synchronises the stream it is given. The enqueueing
 * calls other than mt_scan_rows_noalloc (whose note says nothing on this) may
 * therefore be captured in a CUDA graph and replayed (mt_scan_rows on long
 * rows then records its workspace allocation as a graph node).
 * Calls on different streams, from any host threads, may run concurrently as
 * long as they share no output or scratch buffer.
 *
 * Return codes are mt_status values. A negative code from an enqueueing call
 * means nothing was launched (argument errors) or a CUDA launch failed
 * (MT_ERR_CUDA). Faults that only the device can see (a look-back wait that
 * gave up) are recorded in a device error word and reported by
 * mt_scan_status().
 *
 * Sources, cited by page title and section:
 *   [scan.rs] metaltile-std 0.1.0, src/mlx/scan.rs (Rust kernel DSL page),
 *             module doc "Scan benchmark" and fns mt_scan / mt_scan_exclusive.
 *   [tile]    LuisaCompute, "Tile operations and reductions".
 *   [algos]   Quadrants user guide, "Algorithms".
 */
#ifndef MT_SCAN_H
#define MT_SCAN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MT_F32 = 0,  /* float32 */
    MT_BF16 = 1, /* bfloat16: 8 exponent / 7 fraction bits */
    MT_F16 = 2,  /* IEEE binary16 */
    MT_I32 = 3,  /* int32, two's complement */
    MT_I64 = 4,  /* int64, two's complement */
    MT_U32 = 5,  /* uint32 (1-D scans and reduce) */
    MT_U64 = 6,  /* uint64 (1-D scans and reduce) */
    MT_F64 = 7   /* float64 (1-D scans and reduce) */
} mt_dtype;

/* MT_MUL (product) is a row-scan operation only (mt_scan_rows_op). */
typedef enum { MT_ADD = 0, MT_MIN = 1, MT_MAX = 2, MT_MUL = 3 } mt_op;

typedef enum {
    MT_SCRATCH_SCAN = 1,   /* for mt_exclusive_scan */
    MT_SCRATCH_SELECT = 2, /* for mt_select */
    MT_SCRATCH_REDUCE = 3, /* for mt_reduce */
    MT_SCRATCH_REDUCE_BY_KEY = 4 /* for mt_reduce_by_key_add */
} mt_scratch_kind;

typedef enum {
    MT_OK = 0,
    MT_ERR_ARG = -1,              /* null pointer, negative size, bad enum */
    MT_ERR_DTYPE = -2,            /* dtype not supported by this call */
    MT_ERR_ALIAS = -3,            /* out == arr where in-place is forbidden */
    MT_ERR_CUDA = -4,             /* a CUDA runtime call or launch failed */
    MT_ERR_LOOKBACK_TIMEOUT = -5, /* device: a tile waited too long for a predecessor */
    MT_ERR_ALIGN = -6,            /* pointer not aligned to its element size */
    MT_ERR_TOO_LARGE = -7,        /* needs more than the fixed no-allocation scratch */
    MT_ERR_MEMORY = -8,           /* a pointer the call's kernels cannot reach (see each call) */
    MT_ERR_BOUNDS = -9            /* device, checked build only: an access outside its buffer was skipped */
} mt_status;

/*
 * mt_scan_rows -- sum scan along the last axis of a contiguous row-major
 * [rows, n] tensor.
 *
 * Definition ([scan.rs] module doc "Scan benchmark"; recurrence from [tile]
 * "Why not just infer it from reduce?"): for each row independently,
 *   inclusive: out[r][i] = sum_{j <= i} inp[r][j]
 *   exclusive: out[r][i] = sum_{j <  i} inp[r][j],  out[r][0] = 0.
 * Storage is `dtype` (MT_F32, MT_BF16 or MT_F16) for both inp and out; values
 * are widened to f32, summed in f32 and rounded once to the storage type at
 * the store (round to nearest, ties to even -- [tile] "Storage and
 * arithmetic precision"). The f32 additions may be grouped differently from
 * a left-to-right loop; the element order is never permuted.
 *
 * inp, out : pointers to rows*n elements, each aligned to the element size
 *            (any 16-byte misalignment of a row start is handled). inp == out
 *            (in place) is allowed; other overlaps are not. Device memory,
 *            or -- for rows that fit in one tile (up to about 16384
 *            elements) -- host memory the GPU can reach: pinned host memory
 *            mapped at the same address (cudaHostAlloc / cudaHostRegister
 *            under unified addressing), or any host memory where the device
 *            reads pageable memory (cudaDevAttrPageableMemoryAccess, as on
 *            Grace hosts). The kernels then read and write the host buffers
 *            directly over the host link, with no staging copy. Longer rows
 *            need device memory (their kernel moves data with bulk copies);
 *            other host pointers return MT_ERR_MEMORY.
 * rows, n  : >= 0. rows*n == 0 is a no-op that returns MT_OK.
 * inclusive: nonzero for the inclusive form.
 *
 * Rows longer than one tile are split across CTAs that chain their carries
 * with a single-pass decoupled look-back. Those calls take a small status
 * workspace (128 bytes per tile of 12288 f32 / 16384 bf16 elements, plus 32
 * bytes) from a stream-ordered memory
 * pool owned by the library (cudaMallocFromPoolAsync / cudaFreeAsync on
 * `stream`); rows that fit in one tile use none.
 * Errors: MT_ERR_ARG, MT_ERR_DTYPE, MT_ERR_ALIGN, MT_ERR_MEMORY, MT_ERR_CUDA.
 */
int mt_scan_rows(const void *inp, void *out, int64_t rows, int64_t n, int dtype,
                 int inclusive, void *stream);

/*
 * mt_scan_rows_op -- mt_scan_rows with any of the four operations of the
 * scan.rs page ([scan.rs] "Multi-op scan variants (prod / max / min)"):
 *   op = MT_ADD: sum (identity 0)      -- exactly mt_scan_rows;
 *   op = MT_MUL: product (identity 1.0);
 *   op = MT_MAX: running max (identity -inf);
 *   op = MT_MIN: running min (identity +inf).
 * Inclusive out[r][i] = op(inp[r][0..i]); exclusive out[r][i] =
 * op(inp[r][0..i-1]) with out[r][0] = the identity (stored as +-inf or 1 in
 * the storage type). Values are widened to f32 and combined in f32; sums and
 * products are rounded once to the storage type at the store and may be
 * grouped differently from a left-to-right loop. min keeps the earlier
 * element on ties ((b < a) ? b : a) and max likewise, so min/max results are
 * input values, bit for bit (a zero result carries the sign of the earliest
 * zero). Inputs are assumed NaN-free.
 *
 * Arguments, memory rules, workspace and errors are those of mt_scan_rows;
 * an op outside the four is MT_ERR_ARG.
 */
int mt_scan_rows_op(const void *inp, void *out, int64_t rows, int64_t n, int dtype, int op,
                    int inclusive, void *stream);

/*
 * mt_exclusive_scan -- device-wide exclusive scan of a 1-D array
 * ([algos] "qd.algorithms.exclusive_scan_{add,min,max}"):
 *   out[i] = op(arr[0], ..., arr[i-1]),  out[0] = identity,
 * identity from "Semantics > Common conventions > Identity value": add 0;
 * min +inf (f32) / INT32_MAX / INT64_MAX; max -inf / INT32_MIN / INT64_MIN.
 * Integer add wraps modulo 2^width. min keeps the earlier element on ties
 * ((b < a) ? b : a) and max likewise, so the result is the same for every
 * grouping; f32 add is summed in f32 and may be grouped differently from a
 * left-to-right loop. Inputs are assumed NaN-free (NaN order is unspecified).
 *
 * arr, out : device arrays of `dtype`, aligned to the element size: MT_I32,
 *            MT_I64 or MT_F32, and the other dtypes [algos] lists for its
 *            scans ("qd.algorithms.PrefixSumExecutor": i32, u32, f32, i64,
 *            u64 and f64): MT_U32 and MT_U64 (add wraps; min/max compare as unsigned, identities
 *            UINT_MAX and 0) and MT_F64 (as f32: identities +-inf, earliest
 *            element on ties, sums grouped differently from a left-to-right
 *            loop). out must not be arr ([algos] forbids scanning in place,
 *            "Semantics") -> MT_ERR_ALIAS; other overlaps are undefined.
 * scratch  : device memory of at least
 *            mt_scan_scratch_slots(capacity, dtype, MT_SCRATCH_SCAN) 8-byte
 *            slots, 16-byte aligned. It needs no initialisation ([algos]
 *            "Scratch space"); the call resets what it uses on `stream`.
 *            Concurrent calls must not share one scratch buffer.
 * n_dev    : device pointer to the int32 live count n, read on the device
 *            ([algos] "Key sizing parameters"). n < 0 is treated as 0.
 *            n larger than the capacity the scratch was sized for is
 *            undefined behaviour and is not checked (as on the page).
 * Only out[0:n] is written; out[n:] is left untouched.
 * Two kernels are launched: a status reset and the single-pass scan.
 * Errors: MT_ERR_ARG, MT_ERR_DTYPE, MT_ERR_ALIAS, MT_ERR_ALIGN, MT_ERR_MEMORY (a
 * pointer not in device memory), MT_ERR_CUDA.
 */
int mt_exclusive_scan(const void *arr, void *out, void *scratch, const int32_t *n_dev,
                      int dtype, int op, void *stream);

/*
 * mt_inclusive_scan -- the inclusive form of mt_exclusive_scan:
 *   out[i] = op(arr[0], ..., arr[i])
 * (the left prefix lp[i+1] of [tile] "Why not just infer it from reduce?";
 * [algos] "qd.algorithms.PrefixSumExecutor": arr[i] = sum(arr_original[0..=i]),
 * there for i32 add only and in place). Same dtypes, ops, tie rule,
 * identity, scratch (MT_SCRATCH_SCAN) and live-count rules as
 * mt_exclusive_scan, except that out == arr (in place) is allowed: every
 * tile is read into shared memory before any of it is written.
 * Errors: as mt_exclusive_scan, without MT_ERR_ALIAS.
 */
int mt_inclusive_scan(const void *arr, void *out, void *scratch, const int32_t *n_dev,
                      int dtype, int op, void *stream);

/*
 * mt_reduce -- device-wide reduction ([algos] "qd.algorithms.reduce_{add,min,max}"):
 *   out[0] = op(arr[0], ..., arr[n-1]),  the identity of (op, dtype) for n <= 0.
 * Same dtypes, ops, identities and tie rule as mt_exclusive_scan (for f32
 * min/max the result is the earliest element equal to the extreme, so a zero
 * result carries the sign of the first zero). f32 add is summed in f32 in a
 * fixed grouping (the same bits on every call on the same GPU).
 *
 * arr      : device array of `dtype` (any dtype of mt_exclusive_scan), aligned
 *            to the element size.
 * out      : device pointer to one element of `dtype`.
 * scratch  : device memory of mt_scan_scratch_slots(capacity, dtype,
 *            MT_SCRATCH_REDUCE) 8-byte slots (a fixed size: the header and one
 *            partial per CTA), 8-byte aligned; no initialisation needed.
 * n_dev    : device pointer to the int32 live count n, read on the device.
 * Errors: MT_ERR_ARG, MT_ERR_DTYPE, MT_ERR_ALIGN, MT_ERR_MEMORY (a pointer not
 * in device memory), MT_ERR_CUDA.
 */
int mt_reduce(const void *arr, void *out, void *scratch, const int32_t *n_dev, int dtype, int op,
              void *stream);

/*
 * mt_select -- stream compaction ([algos] "qd.algorithms.select"): every
 * arr[i] with flags[i] == 1 is copied, in input order, into a dense prefix of
 * out, and the number copied is written to *num_out. Elements are 4-byte
 * words copied bit for bit (the copy ignores their type).
 *
 * arr      : device array of n 4-byte elements (4-byte aligned).
 * flags    : device array of n uint8 flags, each exactly 0 or 1 (any other
 *            value is undefined behaviour, as on the page); any alignment.
 *            Flags and values are read in whole 16-byte-aligned blocks, so a
 *            few bytes on either side of each array (in the same 16-byte
 *            blocks, hence the same pages) are read and ignored.
 * out      : device array with room for n elements; only out[0:*num_out] is
 *            written, the rest is left untouched. out must not overlap arr.
 * num_out  : device pointer to one int32.
 * scratch  : mt_scan_scratch_slots(capacity, MT_I32, MT_SCRATCH_SELECT)
 *            8-byte slots, 16-byte aligned, no initialisation needed; not
 *            shared by concurrent calls.
 * n_dev    : device pointer to the int32 live count (n < 0 treated as 0).
 * Errors: MT_ERR_ARG, MT_ERR_ALIAS, MT_ERR_ALIGN, MT_ERR_MEMORY (a pointer not
 * in device memory), MT_ERR_CUDA.
 */
int mt_select(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
              void *scratch, const int32_t *n_dev, void *stream);

/*
 * mt_select_wide -- mt_select for elements of elem_bytes bytes, copied bit
 * for bit: [algos] "qd.algorithms.select" takes no dtype (its scatter moves
 * elements without looking at their type, field by field for structs) and
 * covers 32- and 64-bit scalars and struct element types. elem_bytes is 4,
 * 8, or a struct of 3 to 64 32-bit words (12 to 256 bytes, a multiple of 4;
 * MT_ERR_ARG otherwise). Arguments, scratch (MT_SCRATCH_SELECT), results and
 * errors are those of mt_select; arr and out are aligned to 8 bytes for
 * 8-byte elements and to 4 bytes otherwise (MT_ERR_ALIGN). Struct elements
 * are read straight from arr, only those selected (4- and 8-byte elements
 * are staged through shared memory with the flags).
 */
int mt_select_wide(const void *arr, const uint8_t *flags, void *out, int32_t *num_out,
                   void *scratch, const int32_t *n_dev, int elem_bytes, void *stream);

/*
 * mt_reduce_by_key_add -- run-length sums ([algos]
 * "qd.algorithms.reduce_by_key_add"): every run of consecutive equal keys in
 * keys_in[0:n] becomes one entry, in input order: keys_out[r] = the run's key
 * (that of its first element), values_out[r] = the sum of its values, and
 * *num_runs = the number of runs. Keys equal but separated by other keys form
 * separate runs.
 *
 * keys_in, values_in : device arrays of n elements; key_dtype and
 *            value_dtype are MT_I32, MT_U32 or MT_F32. Float keys compare
 *            with == (each NaN is a run of its own; -0 equals +0). Integer
 *            sums wrap modulo 2^32; f32 sums are added in f32 in a fixed
 *            order (not a left-to-right loop, so not bitwise that loop's).
 *            Both 4-byte aligned and at the same address modulo 16 (they
 *            are read as aligned 16-byte chunks together).
 * keys_out, values_out : device arrays with room for n entries; only the
 *            first *num_runs are written (the page's zero-initialisation of
 *            all of values_out is not done: the tail is untouched).
 * num_runs : device pointer to one int32 (0 for n <= 0).
 * scratch  : mt_scan_scratch_slots(capacity, 0, MT_SCRATCH_REDUCE_BY_KEY)
 *            8-byte slots, 16-byte aligned; no initialisation needed.
 * n_dev    : device pointer to the int32 live count.
 * Errors: MT_ERR_ARG, MT_ERR_DTYPE, MT_ERR_ALIAS (an output is an input),
 * MT_ERR_ALIGN, MT_ERR_MEMORY, MT_ERR_CUDA.
 */
int mt_reduce_by_key_add(const void *keys_in, const void *values_in, void *keys_out, void *values_out,
                         int32_t *num_runs, void *scratch, const int32_t *n_dev, int key_dtype,
                         int value_dtype, void *stream);

/*
 * mt_scan_scratch_slots -- number of 8-byte scratch slots that
 * mt_exclusive_scan / mt_inclusive_scan (kind MT_SCRATCH_SCAN, with their
 * dtype), mt_select / mt_select_wide (kind MT_SCRATCH_SELECT, dtype
 * ignored), mt_reduce (kind MT_SCRATCH_REDUCE, with its dtype; the same size
 * for every capacity) or mt_reduce_by_key_add (kind MT_SCRATCH_REDUCE_BY_KEY,
 * dtype ignored) needs for any live count up to `capacity`. Plain host
 * arithmetic, no device access ([algos] "Scratch space": ask first, then
 * allocate). Returns -1 for a negative capacity or an unknown kind/dtype.
 * The row scans need no scratch argument; the size of the workspace they
 * take themselves is given by mt_scan_rows_scratch_slots.
 */
int64_t mt_scan_scratch_slots(int64_t capacity, int dtype, int kind);

/*
 * mt_scan_rows_scratch_slots -- size, in 8-byte slots, of the look-back
 * workspace that mt_scan_rows / mt_scan_rows_op take from the library's pool
 * and mt_scan_rows_noalloc takes from its fixed array for a [rows, n] call of
 * `dtype` (MT_F32, MT_BF16 or MT_F16), the larger of the two sizes that a row
 * start on a 16-byte boundary or off it needs. 0 when every row fits in one
 * tile (no workspace), -1 for a negative size, another dtype or an overflow.
 * The size depends on both rows and n (each row rounds up to whole tiles), so
 * it is not a kind of mt_scan_scratch_slots, whose sizes follow one capacity.
 * Plain host arithmetic, no device access. A call of mt_scan_rows_noalloc
 * fits its array when this times 8 is at most MT_NOALLOC_SCRATCH_BYTES.
 */
int64_t mt_scan_rows_scratch_slots(int64_t rows, int64_t n, int dtype);

/*
 * mt_scan_status -- synchronise `stream`, then read and clear the device
 * error word of every kernel of the library on the current device.
 * Returns MT_OK, MT_ERR_LOOKBACK_TIMEOUT (a look-back wait gave up and the
 * results of the calls since the last check are not valid), MT_ERR_BOUNDS
 * (only from the bounds-checked build of the library, libmtscan_checked.so:
 * a kernel computed an address outside the buffer it was writing or the
 * shared memory it was using, and skipped that access), or MT_ERR_CUDA.
 * The error words belong to the device, not to a call or a stream: a wait
 * that gave up in a call on any stream of the device is reported to the
 * next mt_scan_status caller on that device, whatever stream it passes (so
 * synchronise the other streams first when their calls must be covered), and
 * that read clears it for everyone.
 */
int mt_scan_status(void *stream);

/* Number of kernels this process has launched through the library (a host
 * counter, for benchmarks that report launch counts). */
uint64_t mt_scan_launches(void);

/* Human-readable name of an mt_status code. */
const char *mt_scan_strerror(int code);

/* 1 in the bounds-checked build of the library (libmtscan_checked.so, whose
 * kernels check every global store and shared-memory access against its
 * buffer and report a bad one as MT_ERR_BOUNDS instead of making it), 0 in
 * the ordinary one. */
int mt_scan_build_checked(void);

/*
 * mt_scan_debug_lookback -- test hook for failure detection. Sets, for the
 * following launches, (a) a global tile index whose CTA computes its results
 * but never publishes its look-back status (-1 = none), and (b) the number of
 * polls after which a waiting tile gives up, records
 * MT_ERR_LOOKBACK_TIMEOUT and publishes its own status so that later tiles
 * are not held (0 = the library default, about a second or more of waiting).
 * Every wait stays bounded. Not for production use.
 */
int mt_scan_debug_lookback(int64_t skip_publish_tile, uint32_t spin_limit);

/*
 * mt_scan_rows_noalloc -- the row scan of mt_scan_rows, for callers that may
 * not allocate device memory. The pages have no counterpart: it exists for
 * programs whose device memory is all reserved up front by another
 * allocator, for loops where an allocation call could take a driver lock or
 * wait on the device, and for hosts that forbid device allocations after
 * start-up. mt_scan_rows takes the look-back records of long rows from a
 * memory pool; this variant takes them from one fixed array inside the
 * library instead, and calls no allocating routine.
 *
 * Arguments, results and the other errors are those of mt_scan_rows, and the
 * look-back test hook (mt_scan_debug_lookback) applies to it as well.
 * Limit: the array holds MT_NOALLOC_SCRATCH_BYTES (1 MiB) on every GPU that
 * loads the library, for the life of the process. A call fits when
 * mt_scan_rows_scratch_slots(rows, n, dtype) * 8 <= MT_NOALLOC_SCRATCH_BYTES;
 * with the library's default tile sizes that is rows * tiles_per_row <= 8191
 * tiles (a tile is 12288 f32 or 16384 bf16/f16 elements of a row; rows that
 * fit one CTA, up to about 16384 elements, use none of it). A larger call
 * returns MT_ERR_TOO_LARGE and launches nothing.
 * The first call that needs the array (rows longer than one tile) in a CUDA
 * context looks up the array's device address in that context (a
 * cudaGetSymbolAddress call, which may load the library's device code), so
 * make that first call before any stream capture. The address is kept per
 * device together with the id of the context it came from and looked up
 * again when another context is current (after cudaDeviceReset, for
 * instance, the next call finds the new context's copy of the array). Every
 * call uses the same array and clears the part it needs first; calls whose
 * kernels overlap on the GPU (different streams, no ordering between them)
 * race on it and must not be made.
 */
#define MT_NOALLOC_SCRATCH_BYTES (1 << 20)
int mt_scan_rows_noalloc(const void *inp, void *out, int64_t rows, int64_t n, int dtype,
                         int inclusive, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MT_SCAN_H */
