/*
 * cpu_allcore.c -- all-core CPU scans, used only as the benchmark's second CPU
 * baseline (next to the single-core oracle). It is not the oracle: the oracle
 * stays plain, single-threaded and fp64. Nothing of the GPU library calls this
 * file, and it shares nothing with it.
 *
 * Row scan. Rows are split into one contiguous block per thread (pthreads); each row is
 * scanned left to right with an f32 running sum -- the accumulation type the
 * metaltile-std scan.rs page ("Scan benchmark") and the GPU path use -- and each
 * output is rounded once to the storage type (round to nearest, ties to even,
 * as in LuisaCompute "Tile operations and reductions", "Storage and arithmetic
 * precision"). Inclusive: out[i] = x[0] + ... + x[i]; exclusive: out[0] = 0,
 * out[i] = x[0] + ... + x[i-1].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { F32 = 0, BF16 = 1, F16 = 2 };

static float bits_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}
static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* bf16 is the top half of an f32. */
static float bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }
static uint16_t f32_to_bf16(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x40u); /* NaN stays NaN (quiet) */
    u += 0x7fffu + ((u >> 16) & 1u);          /* ties to even */
    return (uint16_t)(u >> 16);
}

/* f16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static float f16_to_f32(uint16_t h) {
    const uint32_t s = (uint32_t)(h & 0x8000u) << 16, e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0) { /* zero or subnormal: m * 2^-24, exact in f32 */
        const float v = (float)m * 5.9604644775390625e-08f;
        return bits_f32(f32_bits(v) | s);
    }
    if (e == 31)
        return bits_f32(s | 0x7f800000u | (m << 13));
    return bits_f32(s | ((e + 112u) << 23) | (m << 13));
}
static uint16_t f32_to_f16(float f) {
    const uint32_t u = f32_bits(f);
    const uint16_t s = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u)
        return (uint16_t)(s | 0x7e00u); /* NaN */
    if (a >= 0x477ff000u)               /* 65520 and up round to infinity */
        return (uint16_t)(s | 0x7c00u);
    if (a >= 0x38800000u) {             /* normal in f16 (2^-14 and up) */
        a += 0xfffu + ((a >> 13) & 1u); /* ties to even on the 13 dropped bits */
        return (uint16_t)(s | ((a - 0x38000000u) >> 13));
    }
    /* subnormal or zero in f16: round |f| * 2^24 (exact scaling) to an integer */
    return (uint16_t)(s | (uint16_t)nearbyintf(bits_f32(a) * 16777216.0f));
}

typedef struct {
    const void *in;
    void *out;
    int64_t r0, r1, n;
    int dtype, inclusive;
} job_t;

static void scan_row(const job_t *j, int64_t r) {
    float run = 0.0f;
    if (j->dtype == F32) {
        const float *x = (const float *)j->in + r * j->n;
        float *y = (float *)j->out + r * j->n;
        for (int64_t i = 0; i < j->n; ++i) {
            if (j->inclusive) {
                run += x[i];
                y[i] = run;
            } else {
                y[i] = run;
                run += x[i];
            }
        }
        return;
    }
    const uint16_t *x = (const uint16_t *)j->in + r * j->n;
    uint16_t *y = (uint16_t *)j->out + r * j->n;
    const int b = j->dtype == BF16;
    for (int64_t i = 0; i < j->n; ++i) {
        const float v = b ? bf16_to_f32(x[i]) : f16_to_f32(x[i]);
        if (j->inclusive)
            run += v;
        y[i] = b ? f32_to_bf16(run) : f32_to_f16(run);
        if (!j->inclusive)
            run += v;
    }
}

static void *worker(void *p) {
    const job_t *j = (const job_t *)p;
    for (int64_t r = j->r0; r < j->r1; ++r)
        scan_row(j, r);
    return NULL;
}

/* Scans `rows` rows of `n` elements with `threads` threads (1..256). Returns
 * 0, or -1 for bad arguments or a thread that could not be started. */
int cpu_allcore_scan_rows(const void *in, void *out, int64_t rows, int64_t n, int dtype, int inclusive,
                          int threads) {
    if (rows < 0 || n < 0 || dtype < F32 || dtype > F16 || threads < 1)
        return -1;
    if (threads > 256)
        threads = 256;
    if (threads > rows)
        threads = rows > 0 ? (int)rows : 1;
    job_t jobs[256];
    pthread_t th[256];
    int started = 0, rc = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (job_t){in, out, rows * t / threads, rows * (t + 1) / threads, n, dtype, inclusive != 0};
        if (t > 0) {
            if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) {
                rc = -1;
                break;
            }
            started = t;
        }
    }
    if (rc == 0)
        worker(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    return rc;
}

/*
 * Device-wide exclusive scan of a 1-D array on all cores (Quadrants user guide,
 * "Algorithms", qd.algorithms.exclusive_scan_{add,min,max}): out[0] = identity,
 * out[i] = op(x[0], ..., x[i-1]). The classic two-pass blocked form: each
 * thread folds its contiguous block, one thread scans the block totals, then
 * each thread scans its block again seeded with the total of the blocks before
 * it (two reads of the input, one write). Identities: add 0; min +inf /
 * INT32_MAX / INT64_MAX; max -inf / INT32_MIN / INT64_MIN. Integer add wraps;
 * f32 add runs in f32 (as the GPU path does); min keeps the earlier element on
 * ties ((b < a) ? b : a), max likewise.
 */
enum { I32 = 3, I64 = 4 };
enum { OP_ADD = 0, OP_MIN = 1, OP_MAX = 2 };

typedef union {
    int64_t i;
    float f;
} acc_t;

typedef struct {
    const void *in;
    void *out;
    int64_t b0, b1;
    int dtype, op, pass;
    acc_t seed, total;
} job1d_t;

static acc_t identity1d(int dtype, int op) {
    acc_t a;
    a.i = 0;
    if (dtype == F32) {
        a.f = op == OP_ADD ? 0.0f : (op == OP_MIN ? INFINITY : -INFINITY);
    } else if (dtype == I32) {
        a.i = op == OP_ADD ? 0 : (op == OP_MIN ? INT32_MAX : INT32_MIN);
    } else {
        a.i = op == OP_ADD ? 0 : (op == OP_MIN ? INT64_MAX : INT64_MIN);
    }
    return a;
}

static acc_t combine1d(int dtype, int op, acc_t a, acc_t b) {
    acc_t r;
    if (dtype == F32) {
        r.f = op == OP_ADD ? a.f + b.f : (op == OP_MIN ? (b.f < a.f ? b.f : a.f) : (b.f > a.f ? b.f : a.f));
    } else if (dtype == I32) {
        const int32_t x = (int32_t)a.i, y = (int32_t)b.i;
        r.i = op == OP_ADD ? (int32_t)((uint32_t)x + (uint32_t)y) : (op == OP_MIN ? (y < x ? y : x) : (y > x ? y : x));
    } else {
        r.i = op == OP_ADD ? (int64_t)((uint64_t)a.i + (uint64_t)b.i)
                           : (op == OP_MIN ? (b.i < a.i ? b.i : a.i) : (b.i > a.i ? b.i : a.i));
    }
    return r;
}

static acc_t load1d(int dtype, const void *p, int64_t i) {
    acc_t a;
    if (dtype == F32)
        a.f = ((const float *)p)[i];
    else if (dtype == I32)
        a.i = ((const int32_t *)p)[i];
    else
        a.i = ((const int64_t *)p)[i];
    return a;
}

static void store1d(int dtype, void *p, int64_t i, acc_t a) {
    if (dtype == F32)
        ((float *)p)[i] = a.f;
    else if (dtype == I32)
        ((int32_t *)p)[i] = (int32_t)a.i;
    else
        ((int64_t *)p)[i] = a.i;
}

static void *worker1d(void *p) {
    job1d_t *j = (job1d_t *)p;
    acc_t run = j->pass == 0 ? identity1d(j->dtype, j->op) : j->seed;
    for (int64_t i = j->b0; i < j->b1; ++i) {
        const acc_t x = load1d(j->dtype, j->in, i);
        if (j->pass == 1)
            store1d(j->dtype, j->out, i, run);
        run = combine1d(j->dtype, j->op, run, x);
    }
    j->total = run;
    return NULL;
}

static int run_jobs1d(job1d_t *jobs, int threads) {
    pthread_t th[256];
    int started = 0, rc = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&th[t], NULL, worker1d, &jobs[t]) != 0) {
            rc = -1;
            break;
        }
        started = t;
    }
    if (rc == 0)
        worker1d(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    return rc;
}

/* Exclusive scan of in[0:n] into out[0:n] with `threads` threads (1..256).
 * dtype: 0 f32, 3 i32, 4 i64; op: 0 add, 1 min, 2 max. Returns 0, or -1 for
 * bad arguments or a thread that could not be started. */
int cpu_allcore_exclusive_scan(const void *in, void *out, int64_t n, int dtype, int op, int threads) {
    if (n < 0 || (dtype != F32 && dtype != I32 && dtype != I64) || op < OP_ADD || op > OP_MAX || threads < 1)
        return -1;
    if (threads > 256)
        threads = 256;
    if ((int64_t)threads > n)
        threads = n > 0 ? (int)n : 1;
    job1d_t jobs[256];
    for (int t = 0; t < threads; ++t)
        jobs[t] = (job1d_t){in, out, n * t / threads, n * (t + 1) / threads, dtype, op, 0,
                            identity1d(dtype, op), identity1d(dtype, op)};
    if (run_jobs1d(jobs, threads) != 0)
        return -1;
    acc_t carry = identity1d(dtype, op);
    for (int t = 0; t < threads; ++t) {
        jobs[t].seed = carry;
        jobs[t].pass = 1;
        carry = combine1d(dtype, op, carry, jobs[t].total);
    }
    return run_jobs1d(jobs, threads);
}
