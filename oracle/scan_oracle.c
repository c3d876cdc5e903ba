/*
 * scan_oracle.c -- the CPU oracle for the prefix sum.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the test suite, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes is the plain definition of the scan and nothing else:
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
