// scan_reduce_then_scan.cu -- the three-kernel reduce-then-scan comparison
// path (decoupled look-back paper summary, section 3.2 and Fig. 3; the
// global strategy of the cumsum page, section 1.2):
//   K1  each CTA reduces one tile and writes its aggregate;
//   K2  one CTA turns the aggregates into exclusive tile prefixes, in place;
//   K3  each CTA re-reads its tile and scans it seeded with its prefix
//       (the tile-scan kernel with Lookback::Precomputed).
// About 3n words of global traffic against the single pass's 2n; kept only
// to measure that difference.
#include "scan_device.cuh"

namespace ps {

template <typename T, int THREADS, int ITEMS, bool VEC_IO>
__global__ void __launch_bounds__(THREADS)
tile_reduce_kernel(const T *in, unsigned long long n, typename Traits<T>::U *partials) {
    using Tr = Traits<T>;
    using U = typename Tr::U;
    using V = typename Tr::V;
    constexpr int VEC = Tr::VEC;
    constexpr int ROWS = ITEMS / VEC;
    constexpr int NW = THREADS / 32;
    constexpr long long TILE = (long long)THREADS * ITEMS;
    __shared__ U s_warp[NW];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long tile = blockIdx.x;
    const unsigned long long seg = (unsigned long long)tile * TILE + (unsigned long long)warp * 32 * ITEMS;
    const bool full = (unsigned long long)(tile + 1) * TILE <= n;
    U acc = U(0);
    if (VEC_IO && full) {
        const V *src = reinterpret_cast<const V *>(in + seg) + lane;
        V buf[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) buf[r] = ld_stream(src + r * 32);
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc = acc + (U)vget(buf[r], k);
    } else {
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int k = 0; k < VEC; ++k) {
                const unsigned long long i = seg + (unsigned long long)(r * 32 + lane) * VEC + k;
                if (i < n) acc = acc + (U)in[i];
            }
    }
    acc = warp_sum<U>(acc);
    if (lane == 0) s_warp[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        U t = U(0);
#pragma unroll
        for (int w = 0; w < NW; ++w) t = t + s_warp[w];
        partials[tile] = t;
    }
}

// Exclusive scan of m tile aggregates by one CTA of 1024 threads, in place,
// 1024 values per round with a running carry.
template <typename U>
__global__ void __launch_bounds__(1024) partials_scan_kernel(U *partials, unsigned long long m) {
    __shared__ U s_warp[32];
    __shared__ U s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_carry = U(0);
    __syncthreads();
    for (unsigned long long b = 0; b < m; b += 1024) {
        const unsigned long long i = b + tid;
        const U x = i < m ? partials[i] : U(0);
        const U s = warp_inclusive<U>(x, lane);
        U le = __shfl_up_sync(kFull, s, 1);
        if (lane == 0) le = U(0);
        if (lane == 31) s_warp[warp] = s;
        __syncthreads();
        U wex = U(0), total = U(0);
        for (int w = 0; w < 32; ++w) {
            const U t = s_warp[w];
            if (w < warp) wex = wex + t;
            total = total + t;
        }
        const U carry = s_carry;
        if (i < m) partials[i] = carry + (wex + le);
        __syncthreads();
        if (tid == 0) s_carry = carry + total;
        __syncthreads();
    }
}

template <typename T> constexpr ps_dtype rts_dtype();
template <> constexpr ps_dtype rts_dtype<int32_t>() { return PS_INT32; }
template <> constexpr ps_dtype rts_dtype<int64_t>() { return PS_INT64; }
template <> constexpr ps_dtype rts_dtype<float>() { return PS_FLOAT32; }

template <typename T>
cudaError_t launch_reduce_then_scan(const void *in, void *out, unsigned long long n,
                                    unsigned char *ws, bool exclusive, cudaStream_t s) {
    using U = typename Traits<T>::U;
    constexpr int ITEMS = rts_dtype<T>() == PS_INT64 ? kItems64 : kItems32;
    const size_t tiles = num_tiles(rts_dtype<T>(), n);
    // the partials have a region of their own: the header and the
    // descriptors of the single-pass scans are left as they are
    U *partials = reinterpret_cast<U *>(ws + partials_offset(rts_dtype<T>(), n));
    const T *tin = reinterpret_cast<const T *>(in);
    const bool vec_io = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 15u) == 0;
    cudaError_t e;
    if (vec_io)
        tile_reduce_kernel<T, kThreads, ITEMS, true><<<(unsigned int)tiles, kThreads, 0, s>>>(tin, n, partials);
    else
        tile_reduce_kernel<T, kThreads, ITEMS, false><<<(unsigned int)tiles, kThreads, 0, s>>>(tin, n, partials);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    partials_scan_kernel<U><<<1, 1024, 0, s>>>(partials, tiles);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    PassArgs a{in, out, n, reinterpret_cast<unsigned char *>(partials), nullptr, nullptr, 0, 0};
    return launch_seeded_tile_scan<T>(a, exclusive, s);
}

template cudaError_t launch_reduce_then_scan<int32_t>(const void *, void *, unsigned long long,
                                                      unsigned char *, bool, cudaStream_t);
template cudaError_t launch_reduce_then_scan<int64_t>(const void *, void *, unsigned long long,
                                                      unsigned char *, bool, cudaStream_t);
template cudaError_t launch_reduce_then_scan<float>(const void *, void *, unsigned long long,
                                                    unsigned char *, bool, cudaStream_t);

}  // namespace ps
