// scan_device.cuh -- device building blocks of the single-pass scan:
// value traits, packed tile status descriptors, warp-level scan/reduce and
// the warp-parallel decoupled look-back.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "scan_internal.h"
#include "scan_pipeline.cuh"

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
// Two consecutive 16-byte vectors in one 32-byte store (p 32-byte aligned).
__device__ __forceinline__ void st_stream_pair(ulonglong2 *p, const ulonglong2 &a, const ulonglong2 &b) {
    asm volatile("st.global.cs.v4.u64 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "l"(a.x), "l"(a.y), "l"(b.x), "l"(b.y) : "memory");
}

// ---- tile status descriptors ----------------------------------------------
// Flag and value share one single-copy-atomic 64-bit word, so a reader that
// sees the flag also sees the value and no memory fence is needed
// ("fence-free descriptor updates", section 4.4).  The word also carries the
// epoch (call number) of the call that wrote it; a word from another call
// reads as X, so no call has to reset the descriptors.  For 32-bit values:
//     word = epoch << 34 | flag << 32 | bits(value)
// For 64-bit values two such words are written with one 16-byte store, one
// with the low half and one with the high half of the value, and a reader
// accepts the pair only when both carry the same flag and the current epoch
// (each word is atomic on its own; a torn pair is re-polled).
__device__ __forceinline__ unsigned long long desc_tag(uint32_t flag, uint32_t epoch) {
    return ((unsigned long long)epoch << 34) | ((unsigned long long)flag << 32);
}
__device__ __forceinline__ uint32_t desc_flag(unsigned long long w, uint32_t epoch) {
    return (uint32_t)(w >> 34) == epoch ? (uint32_t)(w >> 32) & 3u : kFlagX;
}

template <typename U, int DW> struct Desc;

template <typename U> struct Desc<U, 1> {
    static __device__ __forceinline__ void store(void *base, long long i, uint32_t flag, U v,
                                                 uint32_t epoch) {
        unsigned long long w = desc_tag(flag, epoch) | to_bits(v);
        unsigned long long *p = reinterpret_cast<unsigned long long *>(
            reinterpret_cast<unsigned char *>(base) + i * kDescStride32);
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(w) : "memory");
    }
    static __device__ __forceinline__ void load(const void *base, long long i, uint32_t epoch,
                                                uint32_t &flag, U &v) {
        const unsigned long long *p = reinterpret_cast<const unsigned long long *>(
            reinterpret_cast<const unsigned char *>(base) + i * kDescStride32);
        unsigned long long w;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
        flag = desc_flag(w, epoch);
        v = from_bits<U>((uint32_t)w);
    }
};

template <> struct Desc<unsigned long long, 2> {
    using U = unsigned long long;
    static __device__ __forceinline__ void store(void *base, long long i, uint32_t flag, U v,
                                                 uint32_t epoch) {
        const unsigned long long t = desc_tag(flag, epoch);
        unsigned long long w0 = t | (v & 0xffffffffull), w1 = t | (v >> 32);
        unsigned long long *p = reinterpret_cast<unsigned long long *>(
            reinterpret_cast<unsigned char *>(base) + i * kDescStride64);
        asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" :: "l"(p), "l"(w0), "l"(w1)
                     : "memory");
    }
    static __device__ __forceinline__ void load(const void *base, long long i, uint32_t epoch,
                                                uint32_t &flag, U &v) {
        const unsigned long long *p = reinterpret_cast<const unsigned long long *>(
            reinterpret_cast<const unsigned char *>(base) + i * kDescStride64);
        unsigned long long w0, w1;
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p)
                     : "memory");
        const uint32_t f0 = desc_flag(w0, epoch), f1 = desc_flag(w1, epoch);
        flag = (f0 == f1) ? f0 : kFlagX;
        v = (w0 & 0xffffffffull) | (w1 << 32);
    }
};

// The producer that takes a tile id fetches that tile's descriptor line into
// L2 at once.  The line was last touched by an earlier call (or never), so
// without this the first look-back poll of it -- and, after an 8-byte
// publish into a line that is not cached, the first read of that partly
// written sector -- goes to DRAM, a round trip of a microsecond or more
// while the memory streams.  By the time the tile publishes A (its data has
// landed) and its successors poll it, the line is in L2.
#ifndef PS_DESC_PREFETCH
#define PS_DESC_PREFETCH 1
#endif
template <int DW>
__device__ __forceinline__ void prefetch_descriptor(const void *desc, long long tile) {
    if (PS_DESC_PREFETCH)
        prefetch_line_l2_last(reinterpret_cast<const unsigned char *>(desc) +
                              tile * (DW == 1 ? kDescStride32 : kDescStride64));
}

// A device-side error of call `epoch` (ps_get_device_status reads it).
__device__ __forceinline__ void report_error(unsigned long long *status, uint32_t epoch,
                                             ps_status code) {
    atomicExch(status, ((unsigned long long)epoch << 8) | (unsigned long long)code);
}

// ---- warp primitives -------------------------------------------------------
// Inclusive Kogge-Stone scan over the 32 lanes with shuffles (the warp scan
// of the cumsum page, section 2, and of the Kogge-Stone network, Fig. 1b of
// the paper summary).  The predecessor's partial is the left operand.
// ---- associative operators ---------------------------------------------------
// combine(a, b) is a (+) b with `a` the earlier part of the sequence; the
// scans only ever combine contiguous parts in that order (section 4.2 of the
// paper summary: non-commutative operators are allowed), and identity() is
// the value of an empty part.  U is the lane type of Traits<T>: integers are
// carried as unsigned bits, so max/min compare them as signed.
__device__ __forceinline__ uint32_t max_of(uint32_t a, uint32_t b) { return (int32_t)a >= (int32_t)b ? a : b; }
__device__ __forceinline__ unsigned long long max_of(unsigned long long a, unsigned long long b) {
    return (long long)a >= (long long)b ? a : b;
}
__device__ __forceinline__ float max_of(float a, float b) { return fmaxf(a, b); }
__device__ __forceinline__ uint32_t min_of(uint32_t a, uint32_t b) { return (int32_t)a <= (int32_t)b ? a : b; }
__device__ __forceinline__ unsigned long long min_of(unsigned long long a, unsigned long long b) {
    return (long long)a <= (long long)b ? a : b;
}
__device__ __forceinline__ float min_of(float a, float b) { return fminf(a, b); }
__device__ __forceinline__ uint32_t lowest_of(uint32_t) { return 0x80000000u; }
__device__ __forceinline__ unsigned long long lowest_of(unsigned long long) { return 0x8000000000000000ull; }
__device__ __forceinline__ float lowest_of(float) { return __int_as_float(0xff800000); }   // -inf
__device__ __forceinline__ uint32_t highest_of(uint32_t) { return 0x7fffffffu; }
__device__ __forceinline__ unsigned long long highest_of(unsigned long long) { return 0x7fffffffffffffffull; }
__device__ __forceinline__ float highest_of(float) { return __int_as_float(0x7f800000); }  // +inf

struct OpSum {
    static constexpr bool kCommutative = true;
    template <typename U> static __device__ __forceinline__ U identity() { return U(0); }
    template <typename U> static __device__ __forceinline__ U combine(U a, U b) { return a + b; }
};
// fp32: fmaxf / fminf, which skip a NaN operand, so the result is the
// maximum (minimum) of the non-NaN elements and the identity when there is
// none; exact, associative and commutative.
struct OpMax {
    static constexpr bool kCommutative = true;
    template <typename U> static __device__ __forceinline__ U identity() { return lowest_of(U()); }
    template <typename U> static __device__ __forceinline__ U combine(U a, U b) { return max_of(a, b); }
};
struct OpMin {
    static constexpr bool kCommutative = true;
    template <typename U> static __device__ __forceinline__ U identity() { return highest_of(U()); }
    template <typename U> static __device__ __forceinline__ U combine(U a, U b) { return min_of(a, b); }
};

// Operators of the two 8-byte pair element types, carried in the int64 lane
// type (the first field in the low 32 bits, the second in the high 32):
//   {int32, fp32} pairs, summed field by field (the int32 field wraps);
//   affine maps x -> a x + b in fp32, {a, b}, composed in sequence order:
//   combine(earlier, later) is "apply earlier, then later",
//       (a1, b1) then (a2, b2) = (a2 a1, a2 b1 + b2),
//   associative but not commutative; the identity is (1, 0).
__device__ __forceinline__ unsigned long long pack2(uint32_t lo, uint32_t hi) {
    return ((unsigned long long)hi << 32) | lo;
}
struct OpPairI32F32 {
    static constexpr bool kCommutative = true;
    template <typename U> static __device__ __forceinline__ U identity() { return U(0); }
    template <typename U> static __device__ __forceinline__ U combine(U a, U b) {
        const uint32_t i = (uint32_t)a + (uint32_t)b;
        const float f = __uint_as_float((uint32_t)(a >> 32)) + __uint_as_float((uint32_t)(b >> 32));
        return pack2(i, __float_as_uint(f));
    }
};
struct OpAffineF32 {
    static constexpr bool kCommutative = false;
    template <typename U> static __device__ __forceinline__ U identity() { return pack2(0x3f800000u, 0u); }
    template <typename U> static __device__ __forceinline__ U combine(U e, U l) {
        const float ea = __uint_as_float((uint32_t)e), eb = __uint_as_float((uint32_t)(e >> 32));
        const float la = __uint_as_float((uint32_t)l), lb = __uint_as_float((uint32_t)(l >> 32));
        return pack2(__float_as_uint(la * ea), __float_as_uint(__fmaf_rn(la, eb, lb)));
    }
};

// Inclusive Kogge-Stone scan over the 32 lanes with shuffles (the warp scan
// of the cumsum page, section 2, and of the Kogge-Stone network, Fig. 1b of
// the paper summary).  The predecessor's partial is the left operand.
template <typename U, typename Op = OpSum> __device__ __forceinline__ U warp_inclusive(U v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        U o = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v = Op::combine(o, v);
    }
    return v;
}

// Reduction over the 32 lanes (butterfly; the operators here are
// commutative, so the lane order does not matter).
template <typename U, typename Op = OpSum> __device__ __forceinline__ U warp_reduce(U v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = Op::combine(v, __shfl_xor_sync(kFull, v, d));
    return v;
}
template <> __device__ __forceinline__ uint32_t warp_reduce<uint32_t, OpSum>(uint32_t v) {
    return __reduce_add_sync(kFull, v);
}
template <> __device__ __forceinline__ uint32_t warp_reduce<uint32_t, OpMax>(uint32_t v) {
    return (uint32_t)__reduce_max_sync(kFull, (int)v);   // signed
}
template <> __device__ __forceinline__ uint32_t warp_reduce<uint32_t, OpMin>(uint32_t v) {
    return (uint32_t)__reduce_min_sync(kFull, (int)v);
}
template <typename U> __device__ __forceinline__ U warp_sum(U v) { return warp_reduce<U, OpSum>(v); }

// Reduction of a look-back window, in which lane l holds the part l places
// before lane 0's: the result, in every lane, is
//     v[31] (+) v[30] (+) ... (+) v[0].
// Commutative operators take the butterfly; the others fold towards lane 0
// with each step's farther (earlier) partial on the left, then broadcast.
template <typename U, typename Op> __device__ __forceinline__ U warp_reduce_window(U v) {
    if constexpr (Op::kCommutative) {
        return warp_reduce<U, Op>(v);
    } else {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const U o = __shfl_down_sync(kFull, v, d);
            if (lane + d < 32) v = Op::combine(o, v);
        }
        return __shfl_sync(kFull, v, 0);
    }
}

// Sleep between polls of a descriptor that is not ready yet.
__device__ __forceinline__ void poll_backoff(uint32_t polls) {
    if (polls > PS_SPIN_POLLS)
        __nanosleep(polls > PS_SLEEP_AFTER_LONG ? PS_SLEEP_NS_LONG : PS_SLEEP_NS_SHORT);
}

// ---- look-back ---------------------------------------------------------------
// Warp-parallel decoupled look-back (section 4.1 step "determine the
// exclusive prefix", in the parallelised form of section 4.4), widened so
// that each lane inspects K consecutive predecessors: position p = lane*K + j
// of the window is tile base - p.  Per round the warp finds the nearest X and
// the nearest P in the window:
//   - an X nearer than every P: re-poll the X descriptors (bounded);
//   - otherwise, a P exists: the values at positions up to and including the
//     nearest P are summed (the segmented reduction with the P tile as the
//     head) and the look-back ends -- X descriptors beyond that P are
//     irrelevant and are not waited for;
//   - otherwise all 32*K are A: they are summed and the window slides back
//     32*K tiles.
// Tiles before tile 0 read as P with the identity; they never decide
// anything because tile 0 only ever publishes P.
//
// A poll cap bounds every wait.  When it is exceeded the status word gets
// PS_ERR_LOOKBACK_TIMEOUT and the missing tiles count as P with the
// identity, so the warp finishes (with a wrong value) instead of hanging.
//
// In a trace build (PS_TRACE) lane 0 writes to *trace, when given, the
// windows walked (high 16 bits) and the re-polls of unpublished
// descriptors (low 16 bits), each saturating; otherwise `trace` is unused.
template <typename U, int DW, int K, typename Op = OpSum>
__device__ __forceinline__ U look_back(const void *desc, long long tile, uint32_t epoch,
                                       uint32_t max_polls, unsigned long long *status,
                                       uint32_t *trace = nullptr) {
    const int lane = threadIdx.x & 31;
    const U ident = Op::template identity<U>();
    U excl = ident;
    long long base = tile - 1;
    uint32_t polls = 0;
    bool gave_up = false;
#ifdef PS_TRACE
    uint32_t windows = 1;
#endif
    while (true) {
        uint32_t f[K];
        U v[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const long long idx = base - (long long)(lane * K + j);
            f[j] = kFlagP;
            v[j] = ident;
            if (idx >= 0) Desc<U, DW>::load(desc, idx, epoch, f[j], v[j]);
        }
        bool done;
        while (true) {
            int px = K, pp = K;   // nearest X / P of this lane (K = none)
#pragma unroll
            for (int j = K - 1; j >= 0; --j) {
                if (f[j] == kFlagX) px = j;
                if (f[j] == kFlagP) pp = j;
            }
            const unsigned mx = __ballot_sync(kFull, px < K);
            const unsigned mp = __ballot_sync(kFull, pp < K);
            int pos_x = 0x7fffffff, pos_p = 0x7fffffff;
            if (mx) {
                const int l = __ffs(mx) - 1;
                pos_x = l * K + __shfl_sync(kFull, px, l);
            }
            if (mp) {
                const int l = __ffs(mp) - 1;
                pos_p = l * K + __shfl_sync(kFull, pp, l);
            }
            if (pos_x < pos_p) {   // a nearer tile has not published yet
                if (++polls > max_polls) {
                    gave_up = true;
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        if (f[j] == kFlagX) { f[j] = kFlagP; v[j] = ident; }
                    continue;
                }
                poll_backoff(polls);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const int pos = lane * K + j;
                    if (f[j] == kFlagX && pos < pos_p)
                        Desc<U, DW>::load(desc, base - (long long)pos, epoch, f[j], v[j]);
                }
                continue;
            }
            // no X before the nearest P (or neither X nor P in the window)
            const int limit = mp ? pos_p : 0x7fffffff;
            U part = ident;
#pragma unroll
            for (int j = K - 1; j >= 0; --j)   // from the farthest tile on: earlier parts on the left
                if (lane * K + j <= limit) part = Op::combine(part, v[j]);
            excl = Op::combine(warp_reduce_window<U, Op>(part), excl);
            done = (mp != 0u);
            break;
        }
        if (done) break;
        base -= 32 * K;
#ifdef PS_TRACE
        ++windows;
#endif
    }
    if (gave_up && lane == 0) report_error(status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
#ifdef PS_TRACE
    if (trace && lane == 0) *trace = (min(windows, 0xffffu) << 16) | min(polls, 0xffffu);
#else
    (void)trace;
#endif
    return excl;
}

// Chained scan (section 3.2 of the paper summary; the adjacent
// synchronisation of the PMPP single-pass page): wait for the immediate
// predecessor's inclusive prefix.  Comparison path only; bounded like the
// look-back.
template <typename U, int DW>
__device__ __forceinline__ U chained_wait(const void *desc, long long tile, uint32_t epoch,
                                          uint32_t max_polls, unsigned long long *status) {
    const int lane = threadIdx.x & 31;
    uint32_t flag = kFlagX;
    U val = U(0);
    uint32_t polls = 0;
    if (lane == 0) {
        Desc<U, DW>::load(desc, tile - 1, epoch, flag, val);
        while (flag != kFlagP) {
            if (++polls > max_polls) {
                report_error(status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                val = U(0);
                break;
            }
            poll_backoff(polls);
            Desc<U, DW>::load(desc, tile - 1, epoch, flag, val);
        }
    }
    return __shfl_sync(kFull, val, 0);
}

// ---- call protocol ----------------------------------------------------------
// Start of a call, by every CTA: the epoch of this call, or false if the
// header is neither fresh (all zero) nor one this library left behind -- a
// workspace that was never zero-filled -- in which case the CTA does nothing
// (ps_get_device_status then reports PS_ERR_WORKSPACE_NOT_INITIALIZED).
__device__ __forceinline__ bool begin_call(const Header *hdr, uint32_t *epoch) {
    const uint32_t magic = *reinterpret_cast<const volatile uint32_t *>(&hdr->magic);
    const uint32_t e = *reinterpret_cast<const volatile uint32_t *>(&hdr->epoch);
    *epoch = e;
    return (magic == kWorkspaceMagic && e <= kEpochMask) || (magic == 0u && e == 0u);
}

// Puts the header back for the next call: tile counter and done count to 0,
// epoch + 1, and the largest size any call declared (the extent an epoch
// wrap clears).
__device__ __forceinline__ void ready_next_call(Header *hdr, unsigned long long ws_bytes, uint32_t epoch) {
    const unsigned long long cap = hdr->capacity > ws_bytes ? hdr->capacity : ws_bytes;
    hdr->capacity = cap;
    hdr->tile_counter = 0ull;
    hdr->done = 0u;
    hdr->epoch = (epoch + 1u) & kEpochMask;
    hdr->magic = kWorkspaceMagic;
}

// The early end of a call, for kernels whose CTAs take their tile ids one
// producer thread each: that thread calls it once, when it takes no more
// ids (past the end, or after a failed wait).  The last of them readies the
// header at once instead of after the last CTA's stores: by then no claim
// of the call is left and every CTA has read the header (each reads it
// before its producer starts), and nothing else of the header is read or
// written during the call but the status word.  Not for the call before an
// epoch wrap, whose clearing of the descriptors needs every CTA done
// (finish_call).
__device__ __forceinline__ void claims_done(Header *hdr, unsigned long long ws_bytes, uint32_t epoch) {
    __threadfence();   // this CTA's last claim precedes its count
    if (atomicAdd(&hdr->done, 1u) == gridDim.x * gridDim.y * gridDim.z - 1) {
        __threadfence();
        ready_next_call(hdr, ws_bytes, epoch);
    }
}

// End of a call, by every thread of every CTA once the CTA's work is done.
// The last CTA to finish (counted with a fenced atomic, so all other CTAs'
// writes precede it) puts the header back for the next call.  When the
// epoch wraps it first clears every descriptor slot the workspace has ever
// been declared to hold, so no descriptor written 2^30 calls ago can pass
// for a current one.  No CTA waits for another here.
__device__ __forceinline__ void finish_call(Header *hdr, unsigned char *ws, unsigned long long ws_bytes,
                                            uint32_t epoch) {
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned int prev = atomicAdd(&hdr->done, 1u);
        s_last = (prev == gridDim.x * gridDim.y * gridDim.z - 1);
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    const unsigned long long cap = hdr->capacity > ws_bytes ? hdr->capacity : ws_bytes;
    if (epoch == kEpochMask) {
        unsigned long long *p = reinterpret_cast<unsigned long long *>(ws + kHeaderBytes);
        const unsigned long long words = (cap - kHeaderBytes) / 8;
        for (unsigned long long i = threadIdx.x; i < words; i += blockDim.x) p[i] = 0ull;
        __threadfence();
        __syncthreads();
    }
    if (threadIdx.x == 0) ready_next_call(hdr, cap, epoch);
}

}  // namespace ps
