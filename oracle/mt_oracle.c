/*
 * CPU oracle for the prefix-scan library -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's shared library. The product path never does, and the
 * two share no code, header, table or helper.
 *
 * It is deliberately plain: one thread, one left-to-right loop per row, float
 * prefixes accumulated in fp64 and rounded once to the output type. Each
 * function names the passage it follows.
 *
 * Sources (web pages, cited by title and section):
 *   [scan.rs]  metaltile-std 0.1.0, src/mlx/scan.rs -- module doc "Scan
 *              benchmark": inclusive out[i] = sum_{j<=i} inp[j]; exclusive
 *              out[i] = sum_{j<i} inp[j] with out[0] = 0; loads and
 *              accumulation in f32, one cast to the storage type at the store.
 *   [tile]     LuisaCompute "Tile operations and reductions":
 *              "Why not just infer it from reduce?" -- the left-prefix
 *              recurrence lp[0] = z, lp[i+1] = op(lp[i], x[i]),
 *              inclusive[i] = lp[i+1], exclusive[i] = lp[i]; scan must not
 *              permute; empty input gives empty output.
 *              "Storage and arithmetic precision" -- bf16 is 8 exponent / 7
 *              fraction bits, half is IEEE binary16 (5 / 10); narrowing
 *              rounds to nearest, ties to even, keeps signed zero and
 *              subnormals, overflows to infinity, quiets NaN.
 *              "Multi-op scan variants (prod / max / min)" -- the same scan
 *              with op x (identity 1.0), max (identity -inf) or min
 *              (identity +inf); the exclusive variant stores the prefix
 *              before the current element.
 *   [algos]    Quadrants "Algorithms" user guide:
 *              "Semantics > Common conventions > Identity value" -- add 0,
 *              min the largest value (+inf, INT_MAX), max the smallest
 *              (-inf, INT_MIN); it seeds exclusive_scan's out[0].
 *              "qd.algorithms.exclusive_scan_{add,min,max}" --
 *              out[i] = op(arr[0:i]).
 *              "qd.algorithms.select" -- copy arr[i] for flags[i] == 1 into a
 *              dense prefix of out in input order; num_out = count; the tail
 *              of out is left untouched.
 *
 * Readings where the pages are silent:
 *   - integer add wraps modulo 2^width (two's complement; unsigned types
 *     likewise); min/max of u32/u64 compare as unsigned, with identities
 *     UINT_MAX (min) and 0 (max);
 *   - f64 add accumulates in long double (at least 64 significand bits);
 *   - min keeps the earlier value on ties: new = (x < acc) ? x : acc, max
 *     likewise with '>'; inputs are NaN-free;
 *   - float add accumulates in fp64 from the decoded storage values.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no -ffast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_I32 = 3, OR_I64 = 4, OR_U32 = 5, OR_U64 = 6, OR_F64 = 7 };
enum { OR_ADD = 0, OR_MIN = 1, OR_MAX = 2, OR_MUL = 3 };

/* ------------------------------------------------------------------------
 * Small-float codecs written from the format definitions ([tile],
 * "Storage and arithmetic precision"). A format has `p` significand bits
 * (hidden bit included), exponent bias `bias` and an all-ones exponent field
 * reserved for infinities and NaNs.
 * ---------------------------------------------------------------------- */

typedef struct {
    int frac_bits;  /* stored fraction bits: bf16 7, half 10 */
    int exp_bits;   /* bf16 8, half 5 */
} small_fmt;

static const small_fmt FMT_BF16 = {7, 8};
static const small_fmt FMT_F16 = {10, 5};

static double small_decode(uint16_t h, small_fmt f)
{
    const int bias = (1 << (f.exp_bits - 1)) - 1;
    const int sign = (h >> (f.frac_bits + f.exp_bits)) & 1;
    const int e = (h >> f.frac_bits) & ((1 << f.exp_bits) - 1);
    const int m = h & ((1 << f.frac_bits) - 1);
    double v;
    if (e == (1 << f.exp_bits) - 1) {
        v = (m == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        /* subnormal: m * 2^(1 - bias - frac_bits) */
        v = ldexp((double)m, 1 - bias - f.frac_bits);
    } else {
        v = ldexp((double)((1 << f.frac_bits) + m), e - bias - f.frac_bits);
    }
    return sign ? -v : v;
}

/* Round a double to the nearest representable value of the format, ties to
 * even, directly from fp64 (one rounding), and return its bit pattern. */
static uint16_t small_encode(double x, small_fmt f)
{
    const int bias = (1 << (f.exp_bits - 1)) - 1;
    const int emin = 1 - bias;                 /* smallest normal exponent */
    const int emax = bias;                     /* largest finite exponent */
    const int p = f.frac_bits + 1;             /* significand bits */
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << (f.frac_bits + f.exp_bits)) : 0;
    const uint16_t exp_all = (uint16_t)(((1u << f.exp_bits) - 1) << f.frac_bits);

    if (isnan(x)) /* quiet NaN: top fraction bit set */
        return (uint16_t)(sign | exp_all | (1u << (f.frac_bits - 1)));
    double a = fabs(x);
    if (isinf(a))
        return (uint16_t)(sign | exp_all);
    if (a == 0.0)
        return sign;

    /* Spacing of representable values at |x|. */
    int e2;
    (void)frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;               /* floor(log2 a) */
    if (E < emin)
        E = emin;                 /* subnormal range: fixed spacing */
    const int q_exp = E - (p - 1);
    double q = ldexp(a, -q_exp);  /* exact: power-of-two scaling */
    double r = nearbyint(q);      /* default mode: to nearest, ties to even */
    double v = ldexp(r, q_exp);   /* the rounded magnitude, exact */

    const double max_finite = ldexp((double)((1 << p) - 1), emax - (p - 1));
    if (v > max_finite)
        return (uint16_t)(sign | exp_all);
    if (v == 0.0) /* below half the smallest subnormal: signed zero */
        return sign;

    /* Encode the exactly representable magnitude v. */
    int ev;
    (void)frexp(v, &ev);
    int Ev = ev - 1;
    if (Ev < emin) {
        /* subnormal: fraction = v / 2^(emin - frac_bits) */
        uint16_t m = (uint16_t)ldexp(v, -(emin - f.frac_bits));
        return (uint16_t)(sign | m);
    }
    uint16_t m = (uint16_t)(ldexp(v, -(Ev - f.frac_bits)) - (double)(1 << f.frac_bits));
    uint16_t efield = (uint16_t)(Ev + bias);
    return (uint16_t)(sign | (uint16_t)(efield << f.frac_bits) | m);
}

double oracle_bf16_to_f64(uint16_t h) { return small_decode(h, FMT_BF16); }
double oracle_f16_to_f64(uint16_t h) { return small_decode(h, FMT_F16); }
uint16_t oracle_f64_to_bf16(double x) { return small_encode(x, FMT_BF16); }
uint16_t oracle_f64_to_f16(double x) { return small_encode(x, FMT_F16); }

/* Vector forms, for the codec pins. */
void oracle_decode_half(const uint16_t *h, double *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = small_decode(h[i], dtype == OR_BF16 ? FMT_BF16 : FMT_F16);
}

void oracle_encode_half(const double *x, uint16_t *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = small_encode(x[i], dtype == OR_BF16 ? FMT_BF16 : FMT_F16);
}

/* Spacing of the format's representable values at the magnitude of v (the
 * "ulp" of a rounded output), using the subnormal gap near zero. */
double oracle_ulp(double v, int dtype)
{
    if (dtype == OR_F32) {
        double a = fabs(v);
        int e2;
        if (a == 0.0)
            return ldexp(1.0, -149);
        (void)frexp(a, &e2);
        int E = e2 - 1;
        if (E < -126)
            E = -126;
        return ldexp(1.0, E - 23);
    }
    small_fmt f = (dtype == OR_BF16) ? FMT_BF16 : FMT_F16;
    const int bias = (1 << (f.exp_bits - 1)) - 1;
    const int emin = 1 - bias;
    double a = fabs(v);
    int E = emin;
    if (a != 0.0) {
        int e2;
        (void)frexp(a, &e2);
        E = e2 - 1;
        if (E < emin)
            E = emin;
    }
    return ldexp(1.0, E - f.frac_bits);
}

static double load_float(const void *base, int64_t i, int dtype)
{
    if (dtype == OR_F32) {
        float v;
        memcpy(&v, (const char *)base + 4 * i, 4);
        return (double)v;
    }
    uint16_t h;
    memcpy(&h, (const char *)base + 2 * i, 2);
    return small_decode(h, dtype == OR_BF16 ? FMT_BF16 : FMT_F16);
}

static void store_float(void *base, int64_t i, double v, int dtype)
{
    if (dtype == OR_F32) {
        float f = (float)v; /* IEEE conversion: round to nearest even */
        memcpy((char *)base + 4 * i, &f, 4);
        return;
    }
    uint16_t h = small_encode(v, dtype == OR_BF16 ? FMT_BF16 : FMT_F16);
    memcpy((char *)base + 2 * i, &h, 2);
}

/* ------------------------------------------------------------------------
 * Row-wise sum scan ([scan.rs] module doc; recurrence from [tile]).
 * Each row of the contiguous [rows, n] input is scanned on its own, left to
 * right, seed 0. `out` receives RN_T of the fp64 prefix. When `prefix64` is
 * non-null it also receives the fp64 prefix itself, and `abs64` the running
 * sum of |x_j| for j <= i (the scale the tolerance is stated against).
 * Returns 0, or -1 on a bad argument.
 * ---------------------------------------------------------------------- */
int oracle_scan_rows(const void *inp, void *out, double *prefix64, double *abs64,
                     int64_t rows, int64_t n, int dtype, int inclusive)
{
    if (rows < 0 || n < 0 || (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F16))
        return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double lp = 0.0;   /* left prefix, seed 0 */
        double mag = 0.0;  /* sum of |x_j| seen so far */
        for (int64_t i = 0; i < n; ++i) {
            const int64_t k = r * n + i;
            const double x = load_float(inp, k, dtype);
            const double lp_next = lp + x;
            mag += fabs(x);
            const double y = inclusive ? lp_next : lp;
            if (out)
                store_float(out, k, y, dtype);
            if (prefix64)
                prefix64[k] = y;
            if (abs64)
                abs64[k] = mag;
            lp = lp_next;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Row-wise scan with any of the page's four operations ([scan.rs] module
 * doc and "Multi-op scan variants (prod / max / min)"; recurrence from
 * [tile]): op = OR_ADD (seed 0), OR_MUL (seed 1.0), OR_MAX (seed -inf) or
 * OR_MIN (seed +inf). Each row is scanned on its own, left to right, in
 * fp64 on the decoded storage values; `out` receives RN_T of the fp64 prefix
 * (min/max prefixes are input values, so they are stored exactly). min keeps
 * the earlier value on ties ((x < lp) ? x : lp), max likewise. When
 * `prefix64` is non-null it receives the fp64 prefix. Returns 0, or -1 on a
 * bad argument.
 * ---------------------------------------------------------------------- */
int oracle_scan_rows_op(const void *inp, void *out, double *prefix64, int64_t rows, int64_t n,
                        int dtype, int op, int inclusive)
{
    if (rows < 0 || n < 0 || (dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_F16) ||
        op < OR_ADD || op > OR_MUL)
        return -1;
    double seed = 0.0;
    if (op == OR_MUL)
        seed = 1.0;
    else if (op == OR_MIN)
        seed = INFINITY;
    else if (op == OR_MAX)
        seed = -INFINITY;
    for (int64_t r = 0; r < rows; ++r) {
        double lp = seed;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t k = r * n + i;
            const double x = load_float(inp, k, dtype);
            double next;
            if (op == OR_ADD)
                next = lp + x;
            else if (op == OR_MUL)
                next = lp * x;
            else if (op == OR_MIN)
                next = (x < lp) ? x : lp;
            else
                next = (x > lp) ? x : lp;
            const double y = inclusive ? next : lp;
            if (out)
                store_float(out, k, y, dtype);
            if (prefix64)
                prefix64[k] = y;
            lp = next;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * The 1-D scans for the unsigned and f64 dtypes that [algos] lists beside
 * i32, i64 and f32 (section "qd.algorithms.PrefixSumExecutor"): the recurrence
 * lp[0] = identity, lp[i+1] = op(lp[i], x[i]); the exclusive form stores
 * lp[i], the inclusive one lp[i+1]. For f64 add, `prefix64` / `abs64` (when
 * non-null) receive the long double prefix rounded to double and the running
 * sum of |x_j| for j <= i.
 * ---------------------------------------------------------------------- */
static void scan_u32(const uint32_t *x, uint32_t *y, int64_t n, int op, int inclusive)
{
    uint32_t lp = (op == OR_MIN) ? UINT32_MAX : 0u;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t next;
        if (op == OR_ADD)
            next = lp + x[i]; /* wraps modulo 2^32 */
        else if (op == OR_MIN)
            next = (x[i] < lp) ? x[i] : lp;
        else
            next = (x[i] > lp) ? x[i] : lp;
        y[i] = inclusive ? next : lp;
        lp = next;
    }
}

static void scan_u64(const uint64_t *x, uint64_t *y, int64_t n, int op, int inclusive)
{
    uint64_t lp = (op == OR_MIN) ? UINT64_MAX : 0u;
    for (int64_t i = 0; i < n; ++i) {
        uint64_t next;
        if (op == OR_ADD)
            next = lp + x[i]; /* wraps modulo 2^64 */
        else if (op == OR_MIN)
            next = (x[i] < lp) ? x[i] : lp;
        else
            next = (x[i] > lp) ? x[i] : lp;
        y[i] = inclusive ? next : lp;
        lp = next;
    }
}

static void scan_f64(const double *x, double *y, double *prefix64, double *abs64, int64_t n, int op,
                     int inclusive)
{
    if (op == OR_ADD) {
        long double lp = 0.0L, mag = 0.0L;
        for (int64_t i = 0; i < n; ++i) {
            const long double next = lp + (long double)x[i];
            mag += fabsl((long double)x[i]);
            const long double v = inclusive ? next : lp;
            if (y)
                y[i] = (double)v;
            if (prefix64)
                prefix64[i] = (double)v;
            if (abs64)
                abs64[i] = (double)mag;
            lp = next;
        }
        return;
    }
    double lp = (op == OR_MIN) ? INFINITY : -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        double next;
        if (op == OR_MIN)
            next = (x[i] < lp) ? x[i] : lp;
        else
            next = (x[i] > lp) ? x[i] : lp;
        y[i] = inclusive ? next : lp;
        lp = next;
    }
}

/* The same dtypes for the scans below; 1 when `dtype` is one of them. */
static int scan_ext(const void *arr, void *out, double *prefix64, double *abs64, int64_t n, int dtype,
                    int op, int inclusive)
{
    if (dtype == OR_U32)
        scan_u32((const uint32_t *)arr, (uint32_t *)out, n, op, inclusive);
    else if (dtype == OR_U64)
        scan_u64((const uint64_t *)arr, (uint64_t *)out, n, op, inclusive);
    else if (dtype == OR_F64)
        scan_f64((const double *)arr, (double *)out, prefix64, abs64, n, op, inclusive);
    else
        return 0;
    return 1;
}

/* ------------------------------------------------------------------------
 * Device-wide exclusive scan ([algos] exclusive_scan_{add,min,max}):
 * out[i] = op(arr[0:i]), out[0] = identity of (op, dtype). Only out[0:n] is
 * written. For f32 add, `out` gets the fp64 prefix rounded to f32 and, when
 * non-null, `prefix64` / `abs64` the fp64 prefix and the running sum of |x_j|
 * for j <= i. Returns 0, or -1 on a bad argument.
 * ---------------------------------------------------------------------- */
int oracle_exclusive_scan(const void *arr, void *out, double *prefix64, double *abs64,
                          int64_t n, int dtype, int op)
{
    if (n < 0 || op < OR_ADD || op > OR_MAX)
        return -1;
    if (scan_ext(arr, out, prefix64, abs64, n, dtype, op, 0))
        return 0;
    if (dtype == OR_I32) {
        const int32_t *x = (const int32_t *)arr;
        int32_t *y = (int32_t *)out;
        if (op == OR_ADD) {
            uint32_t lp = 0; /* unsigned: wraps modulo 2^32 */
            for (int64_t i = 0; i < n; ++i) {
                int32_t v;
                memcpy(&v, &lp, 4);
                y[i] = v;
                lp += (uint32_t)x[i];
            }
        } else {
            int32_t lp = (op == OR_MIN) ? INT32_MAX : INT32_MIN;
            for (int64_t i = 0; i < n; ++i) {
                y[i] = lp;
                if (op == OR_MIN)
                    lp = (x[i] < lp) ? x[i] : lp;
                else
                    lp = (x[i] > lp) ? x[i] : lp;
            }
        }
        return 0;
    }
    if (dtype == OR_I64) {
        const int64_t *x = (const int64_t *)arr;
        int64_t *y = (int64_t *)out;
        if (op == OR_ADD) {
            uint64_t lp = 0; /* wraps modulo 2^64 */
            for (int64_t i = 0; i < n; ++i) {
                int64_t v;
                memcpy(&v, &lp, 8);
                y[i] = v;
                lp += (uint64_t)x[i];
            }
        } else {
            int64_t lp = (op == OR_MIN) ? INT64_MAX : INT64_MIN;
            for (int64_t i = 0; i < n; ++i) {
                y[i] = lp;
                if (op == OR_MIN)
                    lp = (x[i] < lp) ? x[i] : lp;
                else
                    lp = (x[i] > lp) ? x[i] : lp;
            }
        }
        return 0;
    }
    if (dtype == OR_F32) {
        const float *x = (const float *)arr;
        float *y = (float *)out;
        if (op == OR_ADD) {
            double lp = 0.0, mag = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                if (y)
                    y[i] = (float)lp;
                if (prefix64)
                    prefix64[i] = lp;
                mag += fabs((double)x[i]);
                if (abs64)
                    abs64[i] = mag;
                lp += (double)x[i];
            }
        } else {
            float lp = (op == OR_MIN) ? INFINITY : -INFINITY;
            for (int64_t i = 0; i < n; ++i) {
                y[i] = lp;
                if (op == OR_MIN)
                    lp = (x[i] < lp) ? x[i] : lp;
                else
                    lp = (x[i] > lp) ? x[i] : lp;
            }
        }
        return 0;
    }
    return -1;
}

/* ------------------------------------------------------------------------
 * Inclusive form of the device-wide scan: out[i] = op(arr[0..=i]), the left
 * prefix lp[i+1] of the recurrence lp[0] = identity, lp[i+1] = op(lp[i],
 * arr[i]) ([tile] "Why not just infer it from reduce?"; [algos]
 * PrefixSumExecutor: arr[i] = sum(arr_original[0..=i])). Only out[0:n] is
 * written. For f32 add, `out` gets the fp64 prefix rounded to f32 and, when
 * non-null, `prefix64` / `abs64` the fp64 prefix and the running sum of |x_j|
 * for j <= i. Returns 0, or -1 on a bad argument.
 * ---------------------------------------------------------------------- */
int oracle_inclusive_scan(const void *arr, void *out, double *prefix64, double *abs64,
                          int64_t n, int dtype, int op)
{
    if (n < 0 || op < OR_ADD || op > OR_MAX)
        return -1;
    if (scan_ext(arr, out, prefix64, abs64, n, dtype, op, 1))
        return 0;
    if (dtype == OR_I32) {
        const int32_t *x = (const int32_t *)arr;
        int32_t *y = (int32_t *)out;
        if (op == OR_ADD) {
            uint32_t lp = 0; /* unsigned: wraps modulo 2^32 */
            for (int64_t i = 0; i < n; ++i) {
                lp += (uint32_t)x[i];
                int32_t v;
                memcpy(&v, &lp, 4);
                y[i] = v;
            }
        } else {
            int32_t lp = (op == OR_MIN) ? INT32_MAX : INT32_MIN;
            for (int64_t i = 0; i < n; ++i) {
                if (op == OR_MIN)
                    lp = (x[i] < lp) ? x[i] : lp;
                else
                    lp = (x[i] > lp) ? x[i] : lp;
                y[i] = lp;
            }
        }
        return 0;
    }
    if (dtype == OR_I64) {
        const int64_t *x = (const int64_t *)arr;
        int64_t *y = (int64_t *)out;
        if (op == OR_ADD) {
            uint64_t lp = 0; /* wraps modulo 2^64 */
            for (int64_t i = 0; i < n; ++i) {
                lp += (uint64_t)x[i];
                int64_t v;
                memcpy(&v, &lp, 8);
                y[i] = v;
            }
        } else {
            int64_t lp = (op == OR_MIN) ? INT64_MAX : INT64_MIN;
            for (int64_t i = 0; i < n; ++i) {
                if (op == OR_MIN)
                    lp = (x[i] < lp) ? x[i] : lp;
                else
                    lp = (x[i] > lp) ? x[i] : lp;
                y[i] = lp;
            }
        }
        return 0;
    }
    if (dtype == OR_F32) {
        const float *x = (const float *)arr;
        float *y = (float *)out;
        if (op == OR_ADD) {
            double lp = 0.0, mag = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                lp += (double)x[i];
                mag += fabs((double)x[i]);
                if (y)
                    y[i] = (float)lp;
                if (prefix64)
                    prefix64[i] = lp;
                if (abs64)
                    abs64[i] = mag;
            }
        } else {
            float lp = (op == OR_MIN) ? INFINITY : -INFINITY;
            for (int64_t i = 0; i < n; ++i) {
                if (op == OR_MIN)
                    lp = (x[i] < lp) ? x[i] : lp;
                else
                    lp = (x[i] > lp) ? x[i] : lp;
                y[i] = lp;
            }
        }
        return 0;
    }
    return -1;
}

/* ------------------------------------------------------------------------
 * Device-wide reduction ([algos] reduce_{add,min,max}): out[0] =
 * op(arr[0:n]), the identity of (op, dtype) when n == 0 -- the left prefix
 * lp[n] of the same recurrence. For f32 add, out[0] is the fp64 sum rounded
 * to f32 and, when non-null, *sum64 / *abs64 receive the fp64 sum and the sum
 * of |x_j|. Returns 0, or -1 on a bad argument.
 * ---------------------------------------------------------------------- */
int oracle_reduce(const void *arr, void *out, double *sum64, double *abs64, int64_t n, int dtype,
                  int op)
{
    if (n < 0 || op < OR_ADD || op > OR_MAX)
        return -1;
    if (dtype == OR_U32) {
        const uint32_t *x = (const uint32_t *)arr;
        uint32_t r = (op == OR_MIN) ? UINT32_MAX : 0u;
        for (int64_t i = 0; i < n; ++i)
            r = (op == OR_ADD) ? r + x[i] : (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);
        memcpy(out, &r, 4);
        return 0;
    }
    if (dtype == OR_U64) {
        const uint64_t *x = (const uint64_t *)arr;
        uint64_t r = (op == OR_MIN) ? UINT64_MAX : 0u;
        for (int64_t i = 0; i < n; ++i)
            r = (op == OR_ADD) ? r + x[i] : (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);
        memcpy(out, &r, 8);
        return 0;
    }
    if (dtype == OR_F64) {
        const double *x = (const double *)arr;
        double r;
        if (op == OR_ADD) {
            long double acc = 0.0L, mag = 0.0L;
            for (int64_t i = 0; i < n; ++i) {
                acc += (long double)x[i];
                mag += fabsl((long double)x[i]);
            }
            r = (double)acc;
            if (sum64)
                *sum64 = (double)acc;
            if (abs64)
                *abs64 = (double)mag;
        } else {
            r = (op == OR_MIN) ? INFINITY : -INFINITY;
            for (int64_t i = 0; i < n; ++i)
                r = (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);
        }
        memcpy(out, &r, 8);
        return 0;
    }
    if (dtype == OR_I32) {
        const int32_t *x = (const int32_t *)arr;
        int32_t r;
        if (op == OR_ADD) {
            uint32_t acc = 0;
            for (int64_t i = 0; i < n; ++i)
                acc += (uint32_t)x[i];
            memcpy(&r, &acc, 4);
        } else {
            r = (op == OR_MIN) ? INT32_MAX : INT32_MIN;
            for (int64_t i = 0; i < n; ++i)
                r = (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);
        }
        memcpy(out, &r, 4);
        return 0;
    }
    if (dtype == OR_I64) {
        const int64_t *x = (const int64_t *)arr;
        int64_t r;
        if (op == OR_ADD) {
            uint64_t acc = 0;
            for (int64_t i = 0; i < n; ++i)
                acc += (uint64_t)x[i];
            memcpy(&r, &acc, 8);
        } else {
            r = (op == OR_MIN) ? INT64_MAX : INT64_MIN;
            for (int64_t i = 0; i < n; ++i)
                r = (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);
        }
        memcpy(out, &r, 8);
        return 0;
    }
    if (dtype == OR_F32) {
        const float *x = (const float *)arr;
        float r;
        if (op == OR_ADD) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                acc += (double)x[i];
                mag += fabs((double)x[i]);
            }
            r = (float)acc;
            if (sum64)
                *sum64 = acc;
            if (abs64)
                *abs64 = mag;
        } else {
            r = (op == OR_MIN) ? INFINITY : -INFINITY;
            for (int64_t i = 0; i < n; ++i)
                r = (op == OR_MIN) ? ((x[i] < r) ? x[i] : r) : ((x[i] > r) ? x[i] : r);
        }
        memcpy(out, &r, 4);
        return 0;
    }
    return -1;
}

/* ------------------------------------------------------------------------
 * Stream compaction ([algos] select): every arr[i] whose flag is 1 goes to
 * the next slot of out, in input order; the count is returned. Elements are
 * copied as raw 4-byte words (the scatter ignores the element type).
 * out[count:] is not touched.
 * ---------------------------------------------------------------------- */
int64_t oracle_select(const uint32_t *arr, const uint8_t *flags, uint32_t *out, int64_t n)
{
    int64_t j = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (flags[i] == 1) {
            out[j] = arr[i];
            ++j;
        }
    }
    return j;
}

/* ------------------------------------------------------------------------
 * The same compaction for elements of `elem_bytes` bytes, copied byte for
 * byte ([algos] select takes no dtype: its scatter moves elements without
 * looking at their type, field by field for struct elements, so scalars of
 * 4 or 8 bytes and structs of any size are compacted alike).
 * Returns the count, or -1 for elem_bytes < 1.
 * ---------------------------------------------------------------------- */
int64_t oracle_select_wide(const void *arr, const uint8_t *flags, void *out, int64_t n, int elem_bytes)
{
    if (elem_bytes < 1)
        return -1;
    int64_t j = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (flags[i] == 1) {
            memcpy((char *)out + j * elem_bytes, (const char *)arr + i * elem_bytes, (size_t)elem_bytes);
            ++j;
        }
    }
    return j;
}

/* ------------------------------------------------------------------------
 * Reduce by key ([algos] qd.algorithms.reduce_by_key_add): every run of
 * consecutive equal keys becomes one output entry (key, sum of the run's
 * values), in input order; keys equal but separated by other keys form
 * separate runs. Keys and values are i32, u32 or f32 (key_dtype, val_dtype:
 * OR_I32, OR_U32 or OR_F32). Keys compare with == on their type: f32 NaN
 * differs from everything (each NaN is a run of its own) and -0 equals +0.
 * keys_out[r] is the key of the run's first element. Integer sums wrap
 * modulo 2^32; f32 sums accumulate in fp64 and are rounded once; when
 * non-null, sum64 / abs64 receive each run's fp64 sum and sum of |v|.
 * Only the first num_runs entries of the outputs are written. Returns the
 * number of runs, or -1 on a bad argument.
 * ---------------------------------------------------------------------- */
static int key_equal(const void *keys, int64_t i, int64_t j, int key_dtype)
{
    if (key_dtype == OR_F32) {
        float a, b;
        memcpy(&a, (const char *)keys + 4 * i, 4);
        memcpy(&b, (const char *)keys + 4 * j, 4);
        return a == b;
    }
    uint32_t a, b;
    memcpy(&a, (const char *)keys + 4 * i, 4);
    memcpy(&b, (const char *)keys + 4 * j, 4);
    return a == b;
}

int64_t oracle_reduce_by_key_add(const void *keys, const void *vals, void *keys_out, void *vals_out,
                                 double *sum64, double *abs64, int64_t n, int key_dtype, int val_dtype)
{
    if (n < 0 || (key_dtype != OR_I32 && key_dtype != OR_U32 && key_dtype != OR_F32) ||
        (val_dtype != OR_I32 && val_dtype != OR_U32 && val_dtype != OR_F32))
        return -1;
    int64_t r = -1;            /* index of the current run */
    uint32_t isum = 0;         /* integer sum of the current run (wraps) */
    double fsum = 0.0, fabs_sum = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const int head = (i == 0) || !key_equal(keys, i, i - 1, key_dtype);
        if (head) {
            ++r;
            memcpy((char *)keys_out + 4 * r, (const char *)keys + 4 * i, 4);
            isum = 0;
            fsum = 0.0;
            fabs_sum = 0.0;
        }
        if (val_dtype == OR_F32) {
            float v;
            memcpy(&v, (const char *)vals + 4 * i, 4);
            fsum += (double)v;
            fabs_sum += fabs((double)v);
            const float f = (float)fsum;
            memcpy((char *)vals_out + 4 * r, &f, 4);
            if (sum64)
                sum64[r] = fsum;
            if (abs64)
                abs64[r] = fabs_sum;
        } else {
            uint32_t v;
            memcpy(&v, (const char *)vals + 4 * i, 4);
            isum += v;
            memcpy((char *)vals_out + 4 * r, &isum, 4);
        }
    }
    return r + 1;
}
