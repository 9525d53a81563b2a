/*
 * oracle.c -- the sequential CPU oracle for prefix sums and stream compaction.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously correct
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, table or constant with the CUDA sources, and it never calls them.
 *
 * Definitions followed (B. Merry, "Prefix sums on GPUs", GPGPU2 2014, slides
 * "Exclusive Prefix Sum" and "Inclusive Prefix Sum"): for inputs a_0..a_{n-1}
 * and an associative operator (+),
 *     inclusive  s_i = a_0 (+) a_1 (+) ... (+) a_i
 *     exclusive  e_0 = I,  e_i = a_0 (+) ... (+) a_{i-1}
 * Both are computed here as one left-to-right loop per scanned line, exactly
 * as written.  The operators are add, max, min and multiply (the cumulative
 * product that AcceleratedKernels.jl's accumulate API offers as cumprod).
 * Readings where the pages leave a step open:
 *   - exclusive scans take a caller value `init` in place of I and fold it in
 *     on the left of every output (e_i = init (+) a_0 (+) ... (+) a_{i-1});
 *     a missing init means 0 for add and 1 for multiply; max and min have no
 *     neutral element here, so an exclusive max/min without init is refused
 *     (return -2);
 *   - 32- and 64-bit integer add and multiply wrap modulo 2^32 / 2^64 (two's
 *     complement: the low bits of the exact result);
 *   - fp32 and fp64 add and multiply accumulate in fp64 and return fp64 (the
 *     fp64 oracle);
 *   - fp max/min follow C's fmax/fmin: a NaN operand is ignored;
 *   - a (B, R, C) row-major array is scanned along its middle axis: B
 *     independent batches, R scanned positions, C independent lanes.  A 1-D
 *     scan is (1, n, 1); a row scan of a (rows, cols) matrix is (rows, cols,
 *     1); a column scan is (1, rows, cols); an element of L lanes adds L to C.
 *
 * Compaction follows the slides "Other Applications" (compaction: select the
 * objects that satisfy a predicate) and "Atomics" (order must be preserved):
 * the output is the ascending list of indices i with pred(x_i, threshold),
 * the comparison taken in the input's own type.
 *
 * Packing by counts follows the slides "Output Format" and "Solution": object
 * i emits k_i records, the start of its run is the exclusive prefix sum of the
 * counts, and the runs are packed contiguously.  Record r of object i holds
 * the value i.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* Element types, operators and predicates, numbered for the Python wrapper
 * in oracle/__init__.py (its own table; nothing here is shared with the GPU
 * library). */
enum { OR_I32 = 0, OR_U32 = 1, OR_I64 = 2, OR_U64 = 3, OR_F32 = 4, OR_F64 = 5 };
enum { OR_ADD = 0, OR_MAX = 1, OR_MIN = 2, OR_MUL = 3 };
enum { OR_LT = 0, OR_LE = 1, OR_GT = 2, OR_GE = 3, OR_EQ = 4, OR_NE = 5, OR_BITCLR = 6 };

#define OR_OK 0
#define OR_BAD_ARGUMENT (-1)
#define OR_NO_IDENTITY (-2)

/* ---- one operator application per type family ---------------------------- */

static uint32_t op_u32bits_signed(int op, uint32_t acc, uint32_t x)
{
    int32_t a = (int32_t)acc, b = (int32_t)x;
    if (op == OR_ADD) return acc + x; /* modulo 2^32 */
    if (op == OR_MUL) return acc * x; /* the low 32 bits of the product */
    if (op == OR_MAX) return (uint32_t)(a > b ? a : b);
    return (uint32_t)(a < b ? a : b);
}

static uint32_t op_u32bits_unsigned(int op, uint32_t acc, uint32_t x)
{
    if (op == OR_ADD) return acc + x;
    if (op == OR_MUL) return acc * x;
    if (op == OR_MAX) return acc > x ? acc : x;
    return acc < x ? acc : x;
}

static uint64_t op_u64bits_signed(int op, uint64_t acc, uint64_t x)
{
    int64_t a = (int64_t)acc, b = (int64_t)x;
    if (op == OR_ADD) return acc + x; /* modulo 2^64 */
    if (op == OR_MUL) return acc * x; /* the low 64 bits of the product */
    if (op == OR_MAX) return (uint64_t)(a > b ? a : b);
    return (uint64_t)(a < b ? a : b);
}

static uint64_t op_u64bits_unsigned(int op, uint64_t acc, uint64_t x)
{
    if (op == OR_ADD) return acc + x;
    if (op == OR_MUL) return acc * x;
    if (op == OR_MAX) return acc > x ? acc : x;
    return acc < x ? acc : x;
}

static double op_f64(int op, double acc, double x)
{
    if (op == OR_ADD) return acc + x;
    if (op == OR_MUL) return acc * x;
    if (op == OR_MAX) return fmax(acc, x);
    return fmin(acc, x);
}

/* ---- the scans: one sequential loop along the middle axis ---------------- */

/* Index of element (b, r, c) of a row-major (B, R, C) array. */
static int64_t at(int64_t b, int64_t r, int64_t c, int64_t R, int64_t C)
{
    return (b * R + r) * C + c;
}

static void scan_32(int is_signed, int op, int inclusive, const uint32_t *in,
                    uint32_t *out, int64_t B, int64_t R, int64_t C,
                    const uint32_t *init, int64_t init_len)
{
    for (int64_t b = 0; b < B; b++)
        for (int64_t c = 0; c < C; c++) {
            uint32_t acc = op == OR_MUL ? 1u : 0u;
            if (!inclusive && init) acc = init[c % init_len];
            for (int64_t r = 0; r < R; r++) {
                uint32_t x = in[at(b, r, c, R, C)];
                if (inclusive) {
                    if (r == 0) acc = x;
                    else acc = is_signed ? op_u32bits_signed(op, acc, x)
                                         : op_u32bits_unsigned(op, acc, x);
                    out[at(b, r, c, R, C)] = acc;
                } else {
                    out[at(b, r, c, R, C)] = acc;
                    acc = is_signed ? op_u32bits_signed(op, acc, x)
                                    : op_u32bits_unsigned(op, acc, x);
                }
            }
        }
}

static void scan_64(int is_signed, int op, int inclusive, const uint64_t *in,
                    uint64_t *out, int64_t B, int64_t R, int64_t C,
                    const uint64_t *init, int64_t init_len)
{
    for (int64_t b = 0; b < B; b++)
        for (int64_t c = 0; c < C; c++) {
            uint64_t acc = op == OR_MUL ? 1u : 0u;
            if (!inclusive && init) acc = init[c % init_len];
            for (int64_t r = 0; r < R; r++) {
                uint64_t x = in[at(b, r, c, R, C)];
                if (inclusive) {
                    if (r == 0) acc = x;
                    else acc = is_signed ? op_u64bits_signed(op, acc, x)
                                         : op_u64bits_unsigned(op, acc, x);
                    out[at(b, r, c, R, C)] = acc;
                } else {
                    out[at(b, r, c, R, C)] = acc;
                    acc = is_signed ? op_u64bits_signed(op, acc, x)
                                    : op_u64bits_unsigned(op, acc, x);
                }
            }
        }
}

/* Floating point: the input is read as fp64 (exact for fp32) and every
 * partial result is kept in fp64, so `out` is always an fp64 array. */
static void scan_fp(int is_f32, int op, int inclusive, const void *in,
                    double *out, int64_t B, int64_t R, int64_t C,
                    const void *init, int64_t init_len)
{
    for (int64_t b = 0; b < B; b++)
        for (int64_t c = 0; c < C; c++) {
            double acc = op == OR_MUL ? 1.0 : 0.0;
            if (!inclusive && init)
                acc = is_f32 ? (double)((const float *)init)[c % init_len]
                             : ((const double *)init)[c % init_len];
            for (int64_t r = 0; r < R; r++) {
                int64_t i = at(b, r, c, R, C);
                double x = is_f32 ? (double)((const float *)in)[i]
                                  : ((const double *)in)[i];
                if (inclusive) {
                    acc = (r == 0) ? x : op_f64(op, acc, x);
                    out[i] = acc;
                } else {
                    out[i] = acc;
                    acc = op_f64(op, acc, x);
                }
            }
        }
}

/*
 * Scan a row-major (B, R, C) array along its middle axis.
 *   out   int32/uint32 for 32-bit integers, int64/uint64 for 64-bit ones,
 *         fp64 for both float types (see scan_fp).
 *   init  NULL, or init_len elements of the input type; lane c starts from
 *         init[c % init_len].  Used by exclusive scans only.
 * Returns OR_OK, OR_BAD_ARGUMENT or OR_NO_IDENTITY.
 */
int oracle_scan(int dtype, int op, int inclusive, const void *in, void *out,
                int64_t B, int64_t R, int64_t C, const void *init,
                int64_t init_len)
{
    if (B < 0 || R < 0 || C < 0) return OR_BAD_ARGUMENT;
    if (op != OR_ADD && op != OR_MAX && op != OR_MIN && op != OR_MUL) return OR_BAD_ARGUMENT;
    if (init && init_len < 1) return OR_BAD_ARGUMENT;
    if (!inclusive && (op == OR_MAX || op == OR_MIN) && !init) return OR_NO_IDENTITY;
    if (B == 0 || R == 0 || C == 0) return OR_OK;
    switch (dtype) {
    case OR_I32: scan_32(1, op, inclusive, in, out, B, R, C, init, init_len); break;
    case OR_U32: scan_32(0, op, inclusive, in, out, B, R, C, init, init_len); break;
    case OR_I64: scan_64(1, op, inclusive, in, out, B, R, C, init, init_len); break;
    case OR_U64: scan_64(0, op, inclusive, in, out, B, R, C, init, init_len); break;
    case OR_F32: scan_fp(1, op, inclusive, in, out, B, R, C, init, init_len); break;
    case OR_F64: scan_fp(0, op, inclusive, in, out, B, R, C, init, init_len); break;
    default: return OR_BAD_ARGUMENT;
    }
    return OR_OK;
}

/* ---- compaction ---------------------------------------------------------- */

static int holds_f64(int pred, double x, double t)
{
    switch (pred) {
    case OR_LT: return x < t;
    case OR_LE: return x <= t;
    case OR_GT: return x > t;
    case OR_GE: return x >= t;
    case OR_EQ: return x == t;
    default: return x != t;
    }
}

static int holds_f32(int pred, float x, float t)
{
    switch (pred) {
    case OR_LT: return x < t;
    case OR_LE: return x <= t;
    case OR_GT: return x > t;
    case OR_GE: return x >= t;
    case OR_EQ: return x == t;
    default: return x != t;
    }
}

static int holds_i64(int pred, int64_t x, int64_t t)
{
    switch (pred) {
    case OR_LT: return x < t;
    case OR_LE: return x <= t;
    case OR_GT: return x > t;
    case OR_GE: return x >= t;
    case OR_EQ: return x == t;
    default: return x != t;
    }
}

static int holds_u64(int pred, uint64_t x, uint64_t t)
{
    switch (pred) {
    case OR_LT: return x < t;
    case OR_LE: return x <= t;
    case OR_GT: return x > t;
    case OR_GE: return x >= t;
    case OR_EQ: return x == t;
    default: return x != t;
    }
}

/* Does element i satisfy the predicate?  The comparison is made in the
 * element's own type: fp32 data against an fp32 threshold, and so on. */
static int selected(int dtype, int pred, const void *in, int64_t i,
                    const void *threshold)
{
    switch (dtype) {
    case OR_I32: return holds_i64(pred, ((const int32_t *)in)[i], *(const int32_t *)threshold);
    case OR_U32: return holds_u64(pred, ((const uint32_t *)in)[i], *(const uint32_t *)threshold);
    case OR_I64: return holds_i64(pred, ((const int64_t *)in)[i], *(const int64_t *)threshold);
    case OR_U64: return holds_u64(pred, ((const uint64_t *)in)[i], *(const uint64_t *)threshold);
    case OR_F32: return holds_f32(pred, ((const float *)in)[i], *(const float *)threshold);
    default: return holds_f64(pred, ((const double *)in)[i], *(const double *)threshold);
    }
}

/*
 * Stable compaction: out_idx receives, in ascending order, every index i in
 * [0, n) whose element satisfies pred(x_i, *threshold).  out_idx must hold n
 * entries.  Returns the number selected, or a negative error code.
 */
int64_t oracle_compact(int dtype, const void *in, int64_t n, int pred,
                       const void *threshold, int64_t *out_idx)
{
    if (n < 0 || dtype < OR_I32 || dtype > OR_F64) return OR_BAD_ARGUMENT;
    if (pred < OR_LT || pred > OR_NE) return OR_BAD_ARGUMENT;
    int64_t count = 0;
    for (int64_t i = 0; i < n; i++)
        if (selected(dtype, pred, in, i, threshold)) out_idx[count++] = i;
    return count;
}

/* ---- segmented scans -------------------------------------------------------- */

/*
 * Scan restarting at head flags: flags[i] != 0 marks element i as the first of a
 * segment (element 0 always is one).  Inclusive out_i = x_h (+) ... (+) x_i;
 * exclusive out_i = init (+) x_h (+) ... (+) x_{i-1}, out_h = init; h the last
 * head at or before i.  One left-to-right loop that forgets its running value at
 * every head.  Outputs and init typing as for oracle_scan (floats: fp64).
 */
int oracle_scan_segmented(int dtype, int op, int inclusive, const void *in,
                          const uint8_t *flags, void *out, int64_t n,
                          const void *init)
{
    if (n < 0 || dtype < OR_I32 || dtype > OR_F64) return OR_BAD_ARGUMENT;
    if (op != OR_ADD && op != OR_MAX && op != OR_MIN && op != OR_MUL) return OR_BAD_ARGUMENT;
    if (!inclusive && (op == OR_MAX || op == OR_MIN) && !init) return OR_NO_IDENTITY;
    int is_fp = dtype == OR_F32 || dtype == OR_F64;
    int is_signed = dtype == OR_I32 || dtype == OR_I64;
    int wide = dtype == OR_I64 || dtype == OR_U64;
    uint64_t iacc = 0, iinit = op == OR_MUL ? 1u : 0u;
    double facc = 0.0, finit = op == OR_MUL ? 1.0 : 0.0;
    if (init) {
        switch (dtype) {
        case OR_I32: iinit = (uint32_t)*(const int32_t *)init; break;
        case OR_U32: iinit = *(const uint32_t *)init; break;
        case OR_I64: case OR_U64: iinit = *(const uint64_t *)init; break;
        case OR_F32: finit = *(const float *)init; break;
        default: finit = *(const double *)init; break;
        }
    }
    for (int64_t i = 0; i < n; i++) {
        int head = i == 0 || flags[i] != 0;
        double fx = 0.0;
        uint64_t ix = 0;
        switch (dtype) {
        case OR_I32: ix = (uint32_t)((const int32_t *)in)[i]; break;
        case OR_U32: ix = ((const uint32_t *)in)[i]; break;
        case OR_I64: case OR_U64: ix = ((const uint64_t *)in)[i]; break;
        case OR_F32: fx = ((const float *)in)[i]; break;
        default: fx = ((const double *)in)[i]; break;
        }
        if (is_fp) {
            if (!inclusive) ((double *)out)[i] = head ? finit : op_f64(op, finit, facc);
            facc = head ? fx : op_f64(op, facc, fx);
            if (inclusive) ((double *)out)[i] = facc;
        } else if (!wide) {
            uint32_t a = (uint32_t)iacc, x = (uint32_t)ix, t = (uint32_t)iinit;
            uint32_t e = head ? t : (is_signed ? op_u32bits_signed(op, t, a) : op_u32bits_unsigned(op, t, a));
            a = head ? x : (is_signed ? op_u32bits_signed(op, a, x) : op_u32bits_unsigned(op, a, x));
            ((uint32_t *)out)[i] = inclusive ? a : e;
            iacc = a;
        } else {
            uint64_t e = head ? iinit : (is_signed ? op_u64bits_signed(op, iinit, iacc)
                                                   : op_u64bits_unsigned(op, iinit, iacc));
            iacc = head ? ix : (is_signed ? op_u64bits_signed(op, iacc, ix) : op_u64bits_unsigned(op, iacc, ix));
            ((uint64_t *)out)[i] = inclusive ? iacc : e;
        }
    }
    return OR_OK;
}

/* ---- composition of affine maps ----------------------------------------------- */

/*
 * An associative operator that is not commutative, on which the order in which a
 * scan combines its terms shows (The CUDA Handbook, 13.3.4: the packed single-pass
 * descriptor assumes a commutative operator; combining in index order does not).
 * Element i is the affine map f_i(y) = a_i * y + b_i of one integer type, stored as
 * the pair (a_i, b_i) in two consecutive values.  The operator composes two maps in
 * index order, the earlier one applied first:
 *     (a1, b1) (+) (a2, b2) = (a1 * a2,  a2 * b1 + b2),   i.e. y -> f2(f1(y)).
 * Its neutral element is the identity map (1, 0).  Inclusive s_i = f_0 (+) ... (+)
 * f_i, whose b is the value y_i of the first-order linear recurrence
 * y_i = a_i * y_{i-1} + b_i started from y_{-1} = 0; exclusive e_i = init (+) f_0
 * (+) ... (+) f_{i-1} (init NULL: the identity).  32- and 64-bit integers wrap
 * modulo 2^32 / 2^64 (the low bits of the exact results), so signed and unsigned
 * types give the same bits.  One left-to-right loop, as for the other scans.
 * Returns OR_OK or OR_BAD_ARGUMENT (a float type, or n < 0).
 */
int oracle_scan_affine(int dtype, int inclusive, const void *in, void *out, int64_t n,
                       const void *init)
{
    if (n < 0) return OR_BAD_ARGUMENT;
    if (dtype == OR_I32 || dtype == OR_U32) {
        const uint32_t *x = in;
        uint32_t *y = out;
        uint32_t a = 1u, b = 0u;
        if (!inclusive && init) {
            a = ((const uint32_t *)init)[0];
            b = ((const uint32_t *)init)[1];
        }
        for (int64_t i = 0; i < n; i++) {
            uint32_t xa = x[2 * i], xb = x[2 * i + 1];
            if (!inclusive) {
                y[2 * i] = a;
                y[2 * i + 1] = b;
            }
            if (inclusive && i == 0) {
                a = xa;
                b = xb;
            } else {
                uint32_t na = a * xa, nb = xa * b + xb;
                a = na;
                b = nb;
            }
            if (inclusive) {
                y[2 * i] = a;
                y[2 * i + 1] = b;
            }
        }
        return OR_OK;
    }
    if (dtype == OR_I64 || dtype == OR_U64) {
        const uint64_t *x = in;
        uint64_t *y = out;
        uint64_t a = 1u, b = 0u;
        if (!inclusive && init) {
            a = ((const uint64_t *)init)[0];
            b = ((const uint64_t *)init)[1];
        }
        for (int64_t i = 0; i < n; i++) {
            uint64_t xa = x[2 * i], xb = x[2 * i + 1];
            if (!inclusive) {
                y[2 * i] = a;
                y[2 * i + 1] = b;
            }
            if (inclusive && i == 0) {
                a = xa;
                b = xb;
            } else {
                uint64_t na = a * xa, nb = xa * b + xb;
                a = na;
                b = nb;
            }
            if (inclusive) {
                y[2 * i] = a;
                y[2 * i + 1] = b;
            }
        }
        return OR_OK;
    }
    return OR_BAD_ARGUMENT;
}

/* ---- partition ----------------------------------------------------------- */

/* Is bit b of the element's bit pattern clear?  (Integer types.) */
static int bit_clear(int dtype, const void *in, int64_t i, uint64_t b)
{
    uint64_t v;
    switch (dtype) {
    case OR_I32: v = (uint32_t)((const int32_t *)in)[i]; break;
    case OR_U32: v = ((const uint32_t *)in)[i]; break;
    case OR_I64: v = (uint64_t)((const int64_t *)in)[i]; break;
    default: v = ((const uint64_t *)in)[i]; break;
    }
    return ((v >> b) & 1u) == 0;
}

/*
 * Stable partition (slides "Other Applications": partitioning, and the split
 * step of radix sort): out receives first every element that satisfies the
 * predicate, in input order, then every other element, in input order;
 * out_idx[k] is the input index of out[k].  Predicates as for compaction, plus
 * OR_BITCLR for integer types: bit *threshold (as an unsigned bit index) of x
 * is 0.  out holds n elements of the input type, out_idx n entries.  Returns
 * the number selected, or a negative error code.
 */
int64_t oracle_partition(int dtype, const void *in, int64_t n, int pred,
                         const void *threshold, void *out, int64_t *out_idx)
{
    if (n < 0 || dtype < OR_I32 || dtype > OR_F64) return OR_BAD_ARGUMENT;
    if (pred < OR_LT || pred > OR_BITCLR) return OR_BAD_ARGUMENT;
    size_t es = (dtype == OR_I32 || dtype == OR_U32 || dtype == OR_F32) ? 4 : 8;
    uint64_t bit = 0;
    if (pred == OR_BITCLR) {
        if (dtype == OR_F32 || dtype == OR_F64) return OR_BAD_ARGUMENT;
        if (es == 4) bit = *(const uint32_t *)threshold;
        else bit = *(const uint64_t *)threshold;
        if (bit >= 8 * es) return OR_BAD_ARGUMENT;
    }
    int64_t k = 0, m = 0;
    for (int pass = 1; pass >= 0; pass--)   /* the selected ones, then the rest */
        for (int64_t i = 0; i < n; i++) {
            int s = pred == OR_BITCLR ? bit_clear(dtype, in, i, bit)
                                      : selected(dtype, pred, in, i, threshold);
            if (s != pass) continue;
            memcpy((char *)out + k * es, (const char *)in + i * es, es);
            out_idx[k++] = i;
            if (pass) m++;
        }
    return m;
}

/* ---- packing by counts --------------------------------------------------- */

/*
 * Variable-length packing: offsets[i] is the exclusive prefix sum of the
 * counts (in int64, so it never wraps); object i writes the value i into
 * records[offsets[i] .. offsets[i] + k_i), skipping any position at or past
 * `capacity`.  Returns the total number of records (the sum of the counts),
 * or a negative error code when a count is negative.
 */
int64_t oracle_pack_by_counts(const int32_t *counts, int64_t n, int64_t *offsets,
                              int32_t *records, int64_t capacity)
{
    if (n < 0 || capacity < 0) return OR_BAD_ARGUMENT;
    int64_t off = 0;
    for (int64_t i = 0; i < n; i++) {
        if (counts[i] < 0) return OR_BAD_ARGUMENT;
        offsets[i] = off;
        for (int64_t r = 0; r < counts[i]; r++)
            if (off + r < capacity) records[off + r] = (int32_t)i;
        off += counts[i];
    }
    return off;
}
