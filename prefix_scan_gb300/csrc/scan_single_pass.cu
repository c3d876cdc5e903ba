// scan_single_pass.cu -- the single-pass scan kernel (decoupled look-back,
// and the chained variant kept for comparison) and its launcher.
//
// One CTA scans one tile of kThreads * ITEMS consecutive elements:
//   a1  the tile id comes from an atomic counter, not blockIdx, so a CTA
//       only ever waits on tiles whose CTAs are already running (dynamic
//       block index assignment, PMPP single-pass page, section "Dynamic
//       Block Index Assignment"; "virtual processors", section 4.4 of the
//       decoupled look-back paper summary);
//   a2  warp w loads a contiguous 32*ITEMS-element segment with 16-byte
//       loads: row r of the segment is 32 lanes x VEC elements, lane l
//       holding elements r*32*VEC + l*VEC .. +VEC-1 (coalesced);
//   a3  each thread scans its VEC elements of a row sequentially (the
//       serial phase of the three-phase coarsened scan, PMPP
//       work-efficient scan page, "Thread Coarsening");
//   a4  a shuffle-based Kogge-Stone warp scan of the per-lane totals gives
//       each lane its offset within the row; rows are chained in registers;
//   a5  warp totals go through shared memory; each warp sums the totals of
//       the warps before it, and every thread gets the tile aggregate;
//   a6  warp 0 publishes the aggregate (A), or the inclusive prefix (P) for
//       tile 0;
//   a7  warp 0 runs the warp-parallel look-back to get the tile's exclusive
//       prefix;
//   a8  warp 0 publishes the inclusive prefix (P);
//   a9  every thread adds tile prefix + warp offset + row/lane offset and
//       stores its elements with 16-byte streaming stores.
// Steps 1-6 of section 4.1 of the paper summary map to a0 (descriptors of
// earlier calls carry another epoch and read as X; see begin_call and
// finish_call), a1..a5, a6, a7, a8 and a9.
#include "scan_device.cuh"

namespace ps {

#ifndef PS_MIN_BLOCKS
#define PS_MIN_BLOCKS 1
#endif

template <typename T, int THREADS, int ITEMS, bool EXCL, bool VEC_IO, Lookback LB, typename Op>
__global__ void __launch_bounds__(THREADS, PS_MIN_BLOCKS)
single_pass_kernel(PassArgs a) {
    using Tr = Traits<T>;
    using U = typename Tr::U;
    const U ident = Op::template identity<U>();
    using V = typename Tr::V;
    constexpr int VEC = Tr::VEC;
    constexpr int ROWS = ITEMS / VEC;
    constexpr int NW = THREADS / 32;
    constexpr long long TILE = (long long)THREADS * ITEMS;
    static_assert(ITEMS % VEC == 0, "ITEMS must be a multiple of the vector width");

    __shared__ long long s_tile;
    __shared__ U s_warp[NW];
    __shared__ U s_excl;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    Header *hdr = reinterpret_cast<Header *>(a.ws);
    void *desc = a.ws + kHeaderBytes;

    // a1: dynamic tile id
    long long tile;
    uint32_t epoch = 0;
    if (LB == Lookback::Precomputed) {
        tile = blockIdx.x;
    } else {
        // thread 0 alone reads the header (one request per CTA to its line)
        // and, for a workspace it may use, takes the tile id
        __shared__ uint32_t s_epoch;
        __shared__ int s_ok;
        if (tid == 0) {
            uint32_t e;
            s_ok = begin_call(hdr, &e) ? 1 : 0;
            s_epoch = e;
            if (s_ok) s_tile = (long long)atomicAdd(&hdr->tile_counter, 1ull);
        }
        __syncthreads();
        if (!s_ok) return;   // same verdict in every CTA
        epoch = s_epoch;
        tile = s_tile;
    }
    const unsigned long long n = a.n;
    const unsigned long long seg = (unsigned long long)tile * TILE + (unsigned long long)warp * 32 * ITEMS;
    const T *in = reinterpret_cast<const T *>(a.in);
    T *out = reinterpret_cast<T *>(a.out);
    const bool full = (unsigned long long)(tile + 1) * TILE <= n;

    // a2: load
    U v[ROWS][VEC];
    if (VEC_IO && full) {
        const V *src = reinterpret_cast<const V *>(in + seg) + lane;
        V buf[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) buf[r] = ld_stream(src + r * 32);
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) v[r][k] = (U)vget(buf[r], k);
    } else {
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const unsigned long long i = seg + (unsigned long long)(r * 32 + lane) * VEC + k;
                v[r][k] = i < n ? (U)in[i] : ident;
            }
    }

    // a3 + a4: per-thread sequential scan of each row chunk, warp scan of the
    // chunk totals, rows chained in registers.
    U off[ROWS];
    U running = ident;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        U t;
        if (EXCL) {
            U acc = ident;
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const U x = v[r][k];
                v[r][k] = acc;
                acc = Op::combine(acc, x);
            }
            t = acc;
        } else {
#pragma unroll
            for (int k = 1; k < VEC; ++k) v[r][k] = Op::combine(v[r][k - 1], v[r][k]);
            t = v[r][VEC - 1];
        }
        const U s = warp_inclusive<U, Op>(t, lane);
        U le = __shfl_up_sync(kFull, s, 1);
        if (lane == 0) le = ident;
        const U row_total = __shfl_sync(kFull, s, 31);
        off[r] = Op::combine(running, le);
        running = Op::combine(running, row_total);
    }

    // a5: cross-warp scan through shared memory
    if (lane == 0) s_warp[warp] = running;
    __syncthreads();
    U warp_excl = ident, agg = ident;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const U t = s_warp[w];
        if (w < warp) warp_excl = Op::combine(warp_excl, t);
        agg = Op::combine(agg, t);
    }

    // a6..a8: publish, look back, publish
    if (LB == Lookback::Precomputed) {
        // a.ws points at the reduce-then-scan partials for this kernel
        if (tid == 0) s_excl = reinterpret_cast<const U *>(a.ws)[tile];
    } else if (warp == 0) {
        U excl;
        if (tile == 0) {
            // one read of carry_in, by the lane that then publishes tile 0's
            // P: every other tile's P and the write of carry_out follow it,
            // so carry_in may alias carry_out
            U c = ident;
            if (lane == 0 && a.carry_in) c = *reinterpret_cast<const U *>(a.carry_in);
            excl = __shfl_sync(kFull, c, 0);
            if (lane == 0) Desc<U, Tr::DW>::store(desc, 0, kFlagP, Op::combine(excl, agg), epoch);
        } else {
            if (LB == Lookback::Decoupled && lane == 0) Desc<U, Tr::DW>::store(desc, tile, kFlagA, agg, epoch);
            excl = (LB == Lookback::Chained)
                       ? chained_wait<U, Tr::DW>(desc, tile, epoch, a.max_polls, &hdr->status)
                       : look_back<U, Tr::DW, kLookbackK, Op>(desc, tile, epoch, a.max_polls, &hdr->status);
            if (lane == 0) Desc<U, Tr::DW>::store(desc, tile, kFlagP, Op::combine(excl, agg), epoch);
        }
        if (lane == 0) {
            s_excl = excl;
            const long long last = (long long)((n + TILE - 1) / TILE) - 1;
            if (a.carry_out && tile == last) *reinterpret_cast<U *>(a.carry_out) = Op::combine(excl, agg);
        }
    }
    __syncthreads();

    // a9: seeded output
    const U base = Op::combine(s_excl, warp_excl);
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const U o = Op::combine(base, off[r]);
#pragma unroll
        for (int k = 0; k < VEC; ++k) v[r][k] = Op::combine(o, v[r][k]);
    }
    if (VEC_IO && full) {
        V *dst = reinterpret_cast<V *>(out + seg) + lane;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            V w;
#pragma unroll
            for (int k = 0; k < VEC; ++k) vset(w, k, v[r][k]);
            st_stream(dst + r * 32, w);
        }
    } else {
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const unsigned long long i = seg + (unsigned long long)(r * 32 + lane) * VEC + k;
                if (i < n) out[i] = (T)v[r][k];
            }
    }
    if (LB != Lookback::Precomputed) finish_call(hdr, a.ws, a.ws_bytes, epoch);
}

template <typename T> struct ItemsOf { static constexpr int value = kItems32; };
template <> struct ItemsOf<int64_t> { static constexpr int value = kItems64; };

template <typename T, bool EXCL, bool VEC_IO, Lookback LB, typename Op>
cudaError_t launch_variant(const PassArgs &a, size_t tiles, cudaStream_t s) {
    constexpr int ITEMS = ItemsOf<T>::value;
    single_pass_kernel<T, kThreads, ITEMS, EXCL, VEC_IO, LB, Op>
        <<<(unsigned int)tiles, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, bool EXCL, Lookback LB, typename Op = OpSum>
cudaError_t launch_kind(const PassArgs &a, bool vec_io, size_t tiles, cudaStream_t s) {
    return vec_io ? launch_variant<T, EXCL, true, LB, Op>(a, tiles, s)
                  : launch_variant<T, EXCL, false, LB, Op>(a, tiles, s);
}

template <typename T> constexpr ps_dtype dtype_of();
template <> constexpr ps_dtype dtype_of<int32_t>() { return PS_INT32; }
template <> constexpr ps_dtype dtype_of<int64_t>() { return PS_INT64; }
template <> constexpr ps_dtype dtype_of<float>() { return PS_FLOAT32; }

template <typename T, typename Op>
static cudaError_t launch_fallback(const PassArgs &a, bool exclusive, size_t tiles, cudaStream_t s) {
    // one CTA per tile with bounds-checked scalar I/O (arrays not 16-byte aligned)
    return exclusive ? launch_kind<T, true, Lookback::Decoupled, Op>(a, false, tiles, s)
                     : launch_kind<T, false, Lookback::Decoupled, Op>(a, false, tiles, s);
}

template <typename T>
cudaError_t launch_single_pass(const PassArgs &a, bool exclusive, Lookback lb, cudaStream_t s,
                               int op) {
    constexpr ps_dtype dt = dtype_of<T>();
    const size_t tiles = num_tiles(dt, a.n);
    // a0 needs no work here: descriptors of earlier calls carry another
    // epoch and read as X, and the previous call left the counter at 0
    const bool vec_io = ((reinterpret_cast<uintptr_t>(a.in) | reinterpret_cast<uintptr_t>(a.out)) & 15u) == 0;
    if (lb == Lookback::Decoupled) {
        if (a.n <= small_scan_limit<T>()) return launch_small<T>(a, exclusive, op, s);
        if (vec_io) return launch_persistent<T>(a, exclusive, op, s);
        if constexpr (sizeof(T) == 8) {
            if (op == kOpPairI32F32) return launch_fallback<T, OpPairI32F32>(a, exclusive, tiles, s);
            if (op == kOpAffineF32) return launch_fallback<T, OpAffineF32>(a, exclusive, tiles, s);
        }
        switch (op) {
        case kOpMax: return launch_fallback<T, OpMax>(a, exclusive, tiles, s);
        case kOpMin: return launch_fallback<T, OpMin>(a, exclusive, tiles, s);
        default: return launch_fallback<T, OpSum>(a, exclusive, tiles, s);
        }
    }
    return exclusive ? launch_kind<T, true, Lookback::Chained>(a, vec_io, tiles, s)
                     : launch_kind<T, false, Lookback::Chained>(a, vec_io, tiles, s);
}

// The seeded tile scan of the reduce-then-scan comparison path (its third
// kernel) is this kernel with Lookback::Precomputed.
template <typename T>
cudaError_t launch_seeded_tile_scan(const PassArgs &a, bool exclusive, cudaStream_t s) {
    const size_t tiles = num_tiles(dtype_of<T>(), a.n);
    const bool vec_io = ((reinterpret_cast<uintptr_t>(a.in) | reinterpret_cast<uintptr_t>(a.out)) & 15u) == 0;
    return exclusive ? launch_kind<T, true, Lookback::Precomputed>(a, vec_io, tiles, s)
                     : launch_kind<T, false, Lookback::Precomputed>(a, vec_io, tiles, s);
}
template cudaError_t launch_seeded_tile_scan<int32_t>(const PassArgs &, bool, cudaStream_t);
template cudaError_t launch_seeded_tile_scan<int64_t>(const PassArgs &, bool, cudaStream_t);
template cudaError_t launch_seeded_tile_scan<float>(const PassArgs &, bool, cudaStream_t);

template cudaError_t launch_single_pass<int32_t>(const PassArgs &, bool, Lookback, cudaStream_t, int);
template cudaError_t launch_single_pass<int64_t>(const PassArgs &, bool, Lookback, cudaStream_t, int);
template cudaError_t launch_single_pass<float>(const PassArgs &, bool, Lookback, cudaStream_t, int);

// ---- test hook: the look-back alone -----------------------------------------
template <typename T>
__global__ void lookback_probe_kernel(const void *desc, long long tile, uint32_t epoch,
                                      uint32_t max_polls, void *result,
                                      unsigned long long *status) {
    using U = typename Traits<T>::U;
    const U excl = look_back<U, Traits<T>::DW, kLookbackK>(desc, tile, epoch, max_polls, status);
    if (threadIdx.x == 0) *reinterpret_cast<U *>(result) = excl;
}

template <typename T>
cudaError_t launch_lookback_probe(const void *desc, long long tile, uint32_t epoch,
                                  uint32_t max_polls, void *result, unsigned long long *status,
                                  cudaStream_t s) {
    lookback_probe_kernel<T><<<1, 32, 0, s>>>(desc, tile, epoch, max_polls, result, status);
    return cudaGetLastError();
}

template cudaError_t launch_lookback_probe<int32_t>(const void *, long long, uint32_t, uint32_t,
                                                    void *, unsigned long long *, cudaStream_t);
template cudaError_t launch_lookback_probe<int64_t>(const void *, long long, uint32_t, uint32_t,
                                                    void *, unsigned long long *, cudaStream_t);
template cudaError_t launch_lookback_probe<float>(const void *, long long, uint32_t, uint32_t,
                                                  void *, unsigned long long *, cudaStream_t);

}  // namespace ps
