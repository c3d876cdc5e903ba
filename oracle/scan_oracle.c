/*
 * scan_oracle.c -- the CPU oracle for the prefix sum.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the test suite, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes is the plain definition of the scan (and, further down,
 * of stream compaction, running maximum / minimum, reduce-by-key / run-
 * length encoding and the pair scans) and nothing else:
 *
 *   inclusive  y[i] = x[0] + x[1] + ... + x[i]
 *       ("Prefix Sum" definition, page "CUDA-Operators-6-Cumsum", section 1;
 *        problem statement of section 1 of the RTX 4090 scan tutorial page
 *        "smarter.xin/posts/bcb510f9")
 *   exclusive  y[0] = 0,  y[i] = x[0] + ... + x[i-1]
 *       (section "Inclusive 与 Exclusive 的转换" of the same tutorial page)
 *
 * computed by the sequential running sum the cumsum page gives for the CPU
 * (section 1), one element after the other, with no blocking, no reordering
 * and no threads.
 *
 * Readings where the pages are silent:
 *  - Integer overflow: the pages accumulate in a signed int32, whose overflow
 *    is undefined in C.  The sum is taken here in the unsigned type of the
 *    same width, i.e. modulo 2^32 (int32) or 2^64 (int64), and the bits are
 *    stored back unchanged (two's-complement wraparound).
 *  - fp32: accumulated in double and returned in double ("fp64 oracle"); the
 *    caller compares the GPU's fp32 result against it within an error bound
 *    that oracle_abs_prefix_f32 supplies the scale for.
 *  - The exclusive scan is NOT derived from the inclusive one: the running
 *    sum is emitted before the element is added, so "exclusive equals
 *    inclusive shifted by one" is a real check on both.
 *  - n == 0 touches nothing.
 *
 * Parity is pinned by the CPU tests (worked examples printed on the pages,
 * O(n^2) brute force, closed forms, invariants, library cross-checks).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* ---- int32, modulo 2^32 ------------------------------------------------ */

void oracle_inclusive_i32(const int32_t *x, size_t n, int32_t *y)
{
    const uint32_t *xu = (const uint32_t *)x;
    uint32_t *yu = (uint32_t *)y;
    uint32_t sum = 0u;
    for (size_t i = 0; i < n; ++i) {
        sum += xu[i];
        yu[i] = sum;
    }
}

void oracle_exclusive_i32(const int32_t *x, size_t n, int32_t *y)
{
    const uint32_t *xu = (const uint32_t *)x;
    uint32_t *yu = (uint32_t *)y;
    uint32_t sum = 0u;
    for (size_t i = 0; i < n; ++i) {
        uint32_t xi = xu[i]; /* read first: y may alias x */
        yu[i] = sum;
        sum += xi;
    }
}

/* ---- int64, modulo 2^64 ------------------------------------------------ */

void oracle_inclusive_i64(const int64_t *x, size_t n, int64_t *y)
{
    const uint64_t *xu = (const uint64_t *)x;
    uint64_t *yu = (uint64_t *)y;
    uint64_t sum = 0u;
    for (size_t i = 0; i < n; ++i) {
        sum += xu[i];
        yu[i] = sum;
    }
}

void oracle_exclusive_i64(const int64_t *x, size_t n, int64_t *y)
{
    const uint64_t *xu = (const uint64_t *)x;
    uint64_t *yu = (uint64_t *)y;
    uint64_t sum = 0u;
    for (size_t i = 0; i < n; ++i) {
        uint64_t xi = xu[i];
        yu[i] = sum;
        sum += xi;
    }
}

/* ---- fp32 input, fp64 accumulation and result -------------------------- */

void oracle_inclusive_f32(const float *x, size_t n, double *y)
{
    double sum = 0.0;
    for (size_t i = 0; i < n; ++i) {
        sum += (double)x[i];
        y[i] = sum;
    }
}

void oracle_exclusive_f32(const float *x, size_t n, double *y)
{
    double sum = 0.0;
    for (size_t i = 0; i < n; ++i) {
        double xi = (double)x[i];
        y[i] = sum;
        sum += xi;
    }
}

/*
 * Scale of the fp32 error bound: a[i] = |x[0]| + ... + |x[i]| (inclusive) or
 * |x[0]| + ... + |x[i-1]| (exclusive), in double.  The accepted fp32 result
 * satisfies |y[i] - y_fp64[i]| <= 1e-5 * a[i] + 1e-6; the factor is fixed by
 * the test, not here.
 */
void oracle_abs_prefix_f32(const float *x, size_t n, int exclusive, double *a)
{
    double sum = 0.0;
    for (size_t i = 0; i < n; ++i) {
        double xi = (double)x[i];
        if (xi < 0.0)
            xi = -xi;
        if (exclusive) {
            a[i] = sum;
            sum += xi;
        } else {
            sum += xi;
            a[i] = sum;
        }
    }
}

/* ---- stream compaction ("select") and partition -------------------------
 *
 * Decoupled look-back paper summary, section 4.4 ("in-place compaction
 * behaviour"): the output position of a kept element is the exclusive prefix
 * sum of a 0/1 flag array.  The plain definition that this reaches is written
 * out here directly: walk the input once and append every flagged element.
 *
 * select:    out = the elements whose flag is nonzero, in input order;
 *            returns how many.
 * partition: the flagged elements first, in input order, then the others
 *            from the END of `out` backwards (the j-th unflagged element goes
 *            to out[n-1-j]); returns how many were flagged.  Placing the
 *            others from the back is the reading that a single pass can
 *            realise: it needs no total count before writing.
 * Elements are moved as raw 4- or 8-byte words, so int32/fp32 share the
 * 32-bit functions and int64 uses the 64-bit ones.
 */
size_t oracle_select_b32(const uint32_t *x, const uint8_t *flags, size_t n, uint32_t *out)
{
    size_t k = 0;
    for (size_t i = 0; i < n; ++i)
        if (flags[i])
            out[k++] = x[i];
    return k;
}

size_t oracle_select_b64(const uint64_t *x, const uint8_t *flags, size_t n, uint64_t *out)
{
    size_t k = 0;
    for (size_t i = 0; i < n; ++i)
        if (flags[i])
            out[k++] = x[i];
    return k;
}

size_t oracle_partition_b32(const uint32_t *x, const uint8_t *flags, size_t n, uint32_t *out)
{
    size_t k = 0, r = 0;
    for (size_t i = 0; i < n; ++i) {
        if (flags[i])
            out[k++] = x[i];
        else
            out[n - 1 - r++] = x[i];
    }
    return k;
}

size_t oracle_partition_b64(const uint64_t *x, const uint8_t *flags, size_t n, uint64_t *out)
{
    size_t k = 0, r = 0;
    for (size_t i = 0; i < n; ++i) {
        if (flags[i])
            out[k++] = x[i];
        else
            out[n - 1 - r++] = x[i];
    }
    return k;
}

/* Flags from value predicates: op 0 = nonzero, 1 = greater than t,
 * 2 = less than t (IEEE comparisons for fp32: NaN never passes). */
void oracle_flags_i32(const int32_t *x, size_t n, int op, int32_t t, uint8_t *flags)
{
    for (size_t i = 0; i < n; ++i)
        flags[i] = (uint8_t)(op == 0 ? x[i] != 0 : op == 1 ? x[i] > t : x[i] < t);
}

void oracle_flags_i64(const int64_t *x, size_t n, int op, int64_t t, uint8_t *flags)
{
    for (size_t i = 0; i < n; ++i)
        flags[i] = (uint8_t)(op == 0 ? x[i] != 0 : op == 1 ? x[i] > t : x[i] < t);
}

void oracle_flags_f32(const float *x, size_t n, int op, float t, uint8_t *flags)
{
    for (size_t i = 0; i < n; ++i)
        flags[i] = (uint8_t)(op == 0 ? x[i] != 0.0f : op == 1 ? x[i] > t : x[i] < t);
}

/* ---- other associative operators: running maximum / minimum -------------
 *
 * Section 4.2 of the decoupled look-back paper summary: the method applies
 * any associative operator to contiguous parts in order.  The definitions
 * reached, written out directly (op 1 = maximum, 2 = minimum):
 *   inclusive  y[i] = op(x[0], ..., x[i])
 *   exclusive  y[0] = identity, y[i] = op(x[0], ..., x[i-1])
 * with the identity the lowest value of the type for the maximum and the
 * highest for the minimum (INT_MIN / INT_MAX, -inf / +inf).  Integers
 * compare as signed.  fp32 uses fmaxf / fminf, which skip a NaN operand,
 * so a NaN element never becomes the running value.
 */
void oracle_scan_op_i32(const int32_t *x, size_t n, int op, int exclusive, int32_t *y)
{
    int32_t acc = op == 1 ? INT32_MIN : INT32_MAX;
    for (size_t i = 0; i < n; ++i) {
        int32_t xi = x[i];
        if (exclusive)
            y[i] = acc;
        if (op == 1)
            acc = xi > acc ? xi : acc;
        else
            acc = xi < acc ? xi : acc;
        if (!exclusive)
            y[i] = acc;
    }
}

void oracle_scan_op_i64(const int64_t *x, size_t n, int op, int exclusive, int64_t *y)
{
    int64_t acc = op == 1 ? INT64_MIN : INT64_MAX;
    for (size_t i = 0; i < n; ++i) {
        int64_t xi = x[i];
        if (exclusive)
            y[i] = acc;
        if (op == 1)
            acc = xi > acc ? xi : acc;
        else
            acc = xi < acc ? xi : acc;
        if (!exclusive)
            y[i] = acc;
    }
}

void oracle_scan_op_f32(const float *x, size_t n, int op, int exclusive, float *y)
{
    float acc = op == 1 ? -INFINITY : INFINITY;
    for (size_t i = 0; i < n; ++i) {
        float xi = x[i];
        if (exclusive)
            y[i] = acc;
        acc = op == 1 ? fmaxf(acc, xi) : fminf(acc, xi);
        if (!exclusive)
            y[i] = acc;
    }
}

/* ---- reduce-by-key and run-length encoding -------------------------------
 *
 * The paper summary's other single-pass workloads (section A5: reduce-by-key
 * and run-length encoding fused with the scan).  Definitions written out
 * directly: a run is a maximal stretch of consecutive equal keys (keys
 * compared as raw bits, so fp32 keys are equal when their bits are); for
 * every run, in order, the output holds its key and the sum of its values
 * (int32 modulo 2^32; fp32 in double), or, with no values, its length.
 * Returns the number of runs.
 */
size_t oracle_rbk_b32_i32(const uint32_t *keys, const int32_t *vals, size_t n, uint32_t *okeys,
                          int32_t *ovals)
{
    size_t m = 0;
    uint32_t acc = 0u;
    for (size_t i = 0; i < n; ++i) {
        uint32_t v = vals ? (uint32_t)vals[i] : 1u;
        if (i == 0 || keys[i] != keys[i - 1]) {
            if (m > 0)
                ((uint32_t *)ovals)[m - 1] = acc;
            okeys[m++] = keys[i];
            acc = 0u;
        }
        acc += v;
    }
    if (m > 0)
        ((uint32_t *)ovals)[m - 1] = acc;
    return m;
}

size_t oracle_rbk_b64_i32(const uint64_t *keys, const int32_t *vals, size_t n, uint64_t *okeys,
                          int32_t *ovals)
{
    size_t m = 0;
    uint32_t acc = 0u;
    for (size_t i = 0; i < n; ++i) {
        uint32_t v = vals ? (uint32_t)vals[i] : 1u;
        if (i == 0 || keys[i] != keys[i - 1]) {
            if (m > 0)
                ((uint32_t *)ovals)[m - 1] = acc;
            okeys[m++] = keys[i];
            acc = 0u;
        }
        acc += v;
    }
    if (m > 0)
        ((uint32_t *)ovals)[m - 1] = acc;
    return m;
}

/* fp32 values: run sums in double, and the sums of |value| that scale the
 * accepted fp32 error of each run sum. */
size_t oracle_rbk_b32_f32(const uint32_t *keys, const float *vals, size_t n, uint32_t *okeys,
                          double *ovals, double *oabs)
{
    size_t m = 0;
    double acc = 0.0, aacc = 0.0;
    for (size_t i = 0; i < n; ++i) {
        if (i == 0 || keys[i] != keys[i - 1]) {
            if (m > 0) {
                ovals[m - 1] = acc;
                oabs[m - 1] = aacc;
            }
            okeys[m++] = keys[i];
            acc = 0.0;
            aacc = 0.0;
        }
        acc += (double)vals[i];
        aacc += fabs((double)vals[i]);
    }
    if (m > 0) {
        ovals[m - 1] = acc;
        oabs[m - 1] = aacc;
    }
    return m;
}

size_t oracle_rbk_b64_f32(const uint64_t *keys, const float *vals, size_t n, uint64_t *okeys,
                          double *ovals, double *oabs)
{
    size_t m = 0;
    double acc = 0.0, aacc = 0.0;
    for (size_t i = 0; i < n; ++i) {
        if (i == 0 || keys[i] != keys[i - 1]) {
            if (m > 0) {
                ovals[m - 1] = acc;
                oabs[m - 1] = aacc;
            }
            okeys[m++] = keys[i];
            acc = 0.0;
            aacc = 0.0;
        }
        acc += (double)vals[i];
        aacc += fabs((double)vals[i]);
    }
    if (m > 0) {
        ovals[m - 1] = acc;
        oabs[m - 1] = aacc;
    }
    return m;
}

/* ---- scans of 8-byte pair elements ----------------------------------------
 *
 * The paper summary's evaluation data include {int32, fp32} pairs (A4) and
 * section 4.2 allows any associative operator, commutative or not.  Two
 * pair scans, each its plain sequential definition:
 *
 * {int32, fp32} pairs, summed field by field: the int32 field wraps modulo
 * 2^32, the fp32 field is summed in double (with the running sum of |f| that
 * scales the accepted fp32 error).
 */
void oracle_scan_pair_i32_f32(const int32_t *xi, const float *xf, size_t n, int exclusive,
                              int32_t *yi, double *yf, double *yabs)
{
    uint32_t si = 0u;
    double sf = 0.0, sa = 0.0;
    for (size_t k = 0; k < n; ++k) {
        if (exclusive) {
            yi[k] = (int32_t)si;
            yf[k] = sf;
            yabs[k] = sa;
        }
        si += (uint32_t)xi[k];
        sf += (double)xf[k];
        sa += fabs((double)xf[k]);
        if (!exclusive) {
            yi[k] = (int32_t)si;
            yf[k] = sf;
            yabs[k] = sa;
        }
    }
}

/* Affine maps f_k(x) = a_k x + b_k, composed in input order: output k is
 * F_k = f_k o ... o f_0 (exclusive: f_{k-1} o ... o f_0, the identity map
 * for k = 0), F_k(x) = A_k x + B_k, carried in double.  Beside A and B the
 * same recurrence over |a|, |b| gives the magnitudes |A|, sum_j |b_j| prod |a|
 * that scale the accepted fp32 error.  With y_{-1} = 0, B_k is the k-th term
 * of the recurrence y_k = a_k y_{k-1} + b_k. */
void oracle_scan_affine_f32(const float *a, const float *b, size_t n, int exclusive, double *ya,
                            double *yb, double *ya_abs, double *yb_abs)
{
    double A = 1.0, B = 0.0, Aa = 1.0, Ba = 0.0;
    for (size_t k = 0; k < n; ++k) {
        if (exclusive) {
            ya[k] = A;
            yb[k] = B;
            ya_abs[k] = Aa;
            yb_abs[k] = Ba;
        }
        const double ak = (double)a[k], bk = (double)b[k];
        A = ak * A;
        B = ak * B + bk;
        Aa = fabs(ak) * Aa;
        Ba = fabs(ak) * Ba + fabs(bk);
        if (!exclusive) {
            ya[k] = A;
            yb[k] = B;
            ya_abs[k] = Aa;
            yb_abs[k] = Ba;
        }
    }
}
