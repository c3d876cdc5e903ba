// scan_device.cuh -- device building blocks of the single-pass scan:
// value traits, packed tile status descriptors, warp-level scan/reduce and
// the warp-parallel decoupled look-back.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "scan_internal.h"

namespace ps {

constexpr unsigned kFull = 0xffffffffu;

// Status flags of a tile descriptor ("partition descriptor", section 4.1 of
// the decoupled look-back paper summary): X = nothing published yet,
// A = the tile's aggregate is published, P = its inclusive prefix is.
constexpr uint32_t kFlagX = 0, kFlagA = 1, kFlagP = 2;

// ---- value traits ----------------------------------------------------------
// U is the type the additions run in: unsigned integers wrap modulo 2^w
// (two's complement), fp32 stays fp32.  V is the 16-byte vector moved per
// load/store, VEC elements of T.
template <typename T> struct Traits;
template <> struct Traits<int32_t> {
    using U = uint32_t;
    using V = uint4;
    static constexpr int VEC = 4;
    static constexpr int DW = 1;   // descriptor words of 64 bits
};
template <> struct Traits<float> {
    using U = float;
    using V = float4;
    static constexpr int VEC = 4;
    static constexpr int DW = 1;
};
template <> struct Traits<int64_t> {
    using U = unsigned long long;
    using V = ulonglong2;
    static constexpr int VEC = 2;
    static constexpr int DW = 2;
};

__device__ __forceinline__ uint32_t to_bits(uint32_t v) { return v; }
__device__ __forceinline__ uint32_t to_bits(float v) { return __float_as_uint(v); }
template <typename U> __device__ __forceinline__ U from_bits(uint32_t b);
template <> __device__ __forceinline__ uint32_t from_bits<uint32_t>(uint32_t b) { return b; }
template <> __device__ __forceinline__ float from_bits<float>(uint32_t b) { return __uint_as_float(b); }

// Vector element access (the loads/stores move 16 bytes at a time).
__device__ __forceinline__ uint32_t vget(const uint4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ float vget(const float4 &v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
}
__device__ __forceinline__ unsigned long long vget(const ulonglong2 &v, int k) {
    return k == 0 ? v.x : v.y;
}
template <typename V, typename U> __device__ __forceinline__ void vset(V &v, int k, U x);
template <> __device__ __forceinline__ void vset<uint4, uint32_t>(uint4 &v, int k, uint32_t x) {
    if (k == 0) v.x = x; else if (k == 1) v.y = x; else if (k == 2) v.z = x; else v.w = x;
}
template <> __device__ __forceinline__ void vset<float4, float>(float4 &v, int k, float x) {
    if (k == 0) v.x = x; else if (k == 1) v.y = x; else if (k == 2) v.z = x; else v.w = x;
}
template <> __device__ __forceinline__ void vset<ulonglong2, unsigned long long>(
    ulonglong2 &v, int k, unsigned long long x) {
    if (k == 0) v.x = x; else v.y = x;
}

// ---- streaming global memory access --------------------------------------
// Input and output are touched exactly once: evict-first loads and stores
// keep them from displacing the descriptors in L2.
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ld_stream(const float4 *p) {
    float4 v;
    asm volatile("ld.global.cs.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ ulonglong2 ld_stream(const ulonglong2 *p) {
    ulonglong2 v;
    asm volatile("ld.global.cs.v2.u64 {%0,%1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void st_stream(float4 *p, const float4 &v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ void st_stream(ulonglong2 *p, const ulonglong2 &v) {
    asm volatile("st.global.cs.v2.u64 [%0], {%1,%2};" :: "l"(p), "l"(v.x), "l"(v.y) : "memory");
}

// ---- tile status descriptors ----------------------------------------------
// Flag and value share one single-copy-atomic 64-bit word, so a reader that
// sees the flag also sees the value and no memory fence is needed
// ("fence-free descriptor updates", section 4.4).  For 32-bit values:
//     word = flag << 32 | bits(value)
// For 64-bit values two such words are written with one 16-byte store:
//     word0 = flag << 32 | low half,  word1 = flag << 32 | high half
// and a reader accepts the pair only when both flags agree (each word is
// atomic on its own; a torn pair shows differing flags and is re-polled).
template <typename U, int DW> struct Desc;

template <typename U> struct Desc<U, 1> {
    static __device__ __forceinline__ void store(void *base, long long i, uint32_t flag, U v) {
        unsigned long long w = ((unsigned long long)flag << 32) | to_bits(v);
        unsigned long long *p = reinterpret_cast<unsigned long long *>(base) + i;
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(w) : "memory");
    }
    static __device__ __forceinline__ void load(const void *base, long long i, uint32_t &flag, U &v) {
        const unsigned long long *p = reinterpret_cast<const unsigned long long *>(base) + i;
        unsigned long long w;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
        flag = (uint32_t)(w >> 32);
        v = from_bits<U>((uint32_t)w);
    }
};

template <> struct Desc<unsigned long long, 2> {
    using U = unsigned long long;
    static __device__ __forceinline__ void store(void *base, long long i, uint32_t flag, U v) {
        unsigned long long f = (unsigned long long)flag << 32;
        unsigned long long w0 = f | (v & 0xffffffffull), w1 = f | (v >> 32);
        unsigned long long *p = reinterpret_cast<unsigned long long *>(base) + 2 * i;
        asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" :: "l"(p), "l"(w0), "l"(w1)
                     : "memory");
    }
    static __device__ __forceinline__ void load(const void *base, long long i, uint32_t &flag, U &v) {
        const unsigned long long *p = reinterpret_cast<const unsigned long long *>(base) + 2 * i;
        unsigned long long w0, w1;
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p)
                     : "memory");
        uint32_t f0 = (uint32_t)(w0 >> 32), f1 = (uint32_t)(w1 >> 32);
        flag = (f0 == f1) ? f0 : kFlagX;
        v = (w0 & 0xffffffffull) | (w1 << 32);
    }
};

// ---- warp primitives -------------------------------------------------------
// Inclusive Kogge-Stone scan over the 32 lanes with shuffles (the warp scan
// of the cumsum page, section 2, and of the Kogge-Stone network, Fig. 1b of
// the paper summary).  The predecessor's partial is the left operand.
template <typename U> __device__ __forceinline__ U warp_inclusive(U v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        U o = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v = o + v;
    }
    return v;
}

template <typename U> __device__ __forceinline__ U warp_sum(U v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = v + __shfl_xor_sync(kFull, v, d);
    return v;
}
template <> __device__ __forceinline__ uint32_t warp_sum<uint32_t>(uint32_t v) {
    return __reduce_add_sync(kFull, v);
}

// ---- look-back ---------------------------------------------------------------
// Warp-parallel decoupled look-back (section 4.1 step "determine the
// exclusive prefix" with the parallelised form of section 4.4): lane k
// inspects the descriptor of tile base-k.  The warp polls until no lane sees
// X; if some lane sees P, the nearest such tile ends the look-back and the
// values of the tiles from it up to base are summed (the segmented reduction
// with the P tile as head); otherwise all 32 aggregates are summed and the
// window slides back by 32 tiles.  Lanes before tile 0 read as P with the
// identity, which never decides anything because tile 0 only ever publishes
// P.
//
// CHAINED restricts the window to the immediate predecessor and waits for
// its P (the chained scan of section 3.2; comparison path only).
//
// A poll cap bounds every wait.  When it is exceeded the status word gets
// PS_ERR_LOOKBACK_TIMEOUT and still-missing tiles count as P with the
// identity, so the warp finishes (with a wrong value) instead of hanging.
template <typename U, int DW, bool CHAINED>
__device__ __forceinline__ U look_back(const void *desc, long long tile, uint32_t max_polls,
                                       unsigned int *status) {
    const int lane = threadIdx.x & 31;
    U excl = U(0);
    long long base = tile - 1;
    uint32_t polls = 0;
    bool gave_up = false;
    while (true) {
        const long long idx = base - lane;
        const bool active = CHAINED ? (lane == 0) : true;
        uint32_t flag = kFlagP;
        U val = U(0);
        if (active && idx >= 0) Desc<U, DW>::load(desc, idx, flag, val);
        // poll until every inspected tile has published something
        // (CHAINED: until the predecessor has published its prefix)
        unsigned pending;
        while ((pending = __ballot_sync(kFull, CHAINED ? (flag != kFlagP) : (flag == kFlagX))) != 0u) {
            if (++polls > max_polls) {
                gave_up = true;
                if (pending & (1u << lane)) { flag = kFlagP; val = U(0); }
                break;
            }
            if (polls > 8) __nanosleep(polls > 64 ? 512 : 32);
            if (pending & (1u << lane)) Desc<U, DW>::load(desc, idx, flag, val);
        }
        const unsigned pmask = __ballot_sync(kFull, flag == kFlagP);
        if (pmask != 0u) {
            const int first = __ffs(pmask) - 1;
            excl = warp_sum<U>(lane <= first ? val : U(0)) + excl;
            break;
        }
        excl = warp_sum<U>(val) + excl;
        base -= 32;
    }
    if (gave_up && lane == 0) atomicMax(status, (unsigned int)PS_ERR_LOOKBACK_TIMEOUT);
    return excl;
}

}  // namespace ps
