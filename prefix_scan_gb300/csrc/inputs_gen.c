/*
 * inputs_gen.c -- seeded synthetic input fill (host, plain C).
 *
 * The counter-based generator documented in prefix_scan_gb300/inputs.py:
 * element i of the stream keyed by `key` is
 *     splitmix64_mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 * with the SplitMix64 output function (Steele, Lea & Flood, OOPSLA 2014).
 * This file only produces input values; it contains no scan arithmetic and
 * is shared by the test/bench harness on both sides of a parity check.
 */
#include <stddef.h>
#include <stdint.h>

#define GEN_GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t gen_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t gen_at(uint64_t key, uint64_t i)
{
    return gen_mix(key + (i + 1u) * GEN_GOLDEN);
}

void gen_hash_u64(uint64_t key, uint64_t start, size_t count, uint64_t *out)
{
    for (size_t k = 0; k < count; ++k)
        out[k] = gen_at(key, start + k);
}

/* lo + (((h >> 32) * span) >> 32), span in [1, 2^32] */
void gen_uniform_i32(uint64_t key, uint64_t start, size_t count, int64_t lo, uint64_t span,
                     int32_t *out)
{
    for (size_t k = 0; k < count; ++k) {
        uint64_t h = gen_at(key, start + k);
        int64_t v = lo + (int64_t)(((h >> 32) * span) >> 32);
        out[k] = (int32_t)v;
    }
}

void gen_uniform_i64(uint64_t key, uint64_t start, size_t count, int64_t lo, uint64_t span,
                     int64_t *out)
{
    for (size_t k = 0; k < count; ++k) {
        uint64_t h = gen_at(key, start + k);
        out[k] = lo + (int64_t)(((h >> 32) * span) >> 32);
    }
}

/* Bernoulli(1/2): the top bit of the hash. elem_size 4 (int32) or 8 (int64). */
void gen_bernoulli(uint64_t key, uint64_t start, size_t count, int elem_size, void *out)
{
    if (elem_size == 8) {
        int64_t *o = (int64_t *)out;
        for (size_t k = 0; k < count; ++k)
            o[k] = (int64_t)(gen_at(key, start + k) >> 63);
    } else {
        int32_t *o = (int32_t *)out;
        for (size_t k = 0; k < count; ++k)
            o[k] = (int32_t)(gen_at(key, start + k) >> 63);
    }
}

/* fp32 on the grid (h >> 40) * 2^-23 - 1, exact in fp32. */
void gen_uniform_f32(uint64_t key, uint64_t start, size_t count, float *out)
{
    for (size_t k = 0; k < count; ++k) {
        uint64_t h = gen_at(key, start + k);
        out[k] = (float)((double)(h >> 40) * (1.0 / 8388608.0) - 1.0);
    }
}

/* Full-range int32: the low 32 bits of the hash. */
void gen_full_i32(uint64_t key, uint64_t start, size_t count, int32_t *out)
{
    uint32_t *o = (uint32_t *)out;
    for (size_t k = 0; k < count; ++k)
        o[k] = (uint32_t)gen_at(key, start + k);
}
