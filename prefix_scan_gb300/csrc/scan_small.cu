// scan_small.cu -- the scan of a short array (at most two tiles) in one CTA.
//
// For n up to 2 x 8192 (32-bit types) or 2 x 4096 (int64 and the pair
// types) the whole array fits one CTA's registers, so no tile needs a
// predecessor's prefix: 1024 threads load it in rows of 16-byte vectors,
// scan each row (each thread its vector serially, a shuffle Kogge-Stone
// warp scan of the thread totals, then one warp scans the 32 warp totals
// -- the three-phase block scan of the PMPP work-efficient scan page,
// "Thread Coarsening"), chain the rows, and store.  No atomic, descriptor
// or end-of-call hand-off: the call costs one launch and one round trip to
// memory instead of the persistent kernel's chain of dependent ones
// (tile-id atomic, bulk copy, aggregate, hand-offs, end-of-call counter).
//
// It reads the workspace header only to keep the workspace contract: a
// workspace that was never zero-filled makes it do nothing, as it does the
// other kernels.  It leaves the header (tile counter, call number)
// untouched.
#include "scan_device.cuh"

namespace ps {

namespace {

constexpr int kSmallThreads = 1024;
constexpr int kSmallRows = 4;   // rows of kSmallThreads vectors

}  // namespace

template <typename T>
constexpr unsigned long long small_scan_max() {
    return (unsigned long long)kSmallRows * kSmallThreads * Traits<T>::VEC;
}

template <typename T, bool EXCL, typename Op>
__global__ void __launch_bounds__(kSmallThreads, 1) small_scan_kernel(PassArgs a, int vec_io) {
    using Tr = Traits<T>;
    using U = typename Tr::U;
    using V = typename Tr::V;
    constexpr int VEC = Tr::VEC;
    constexpr int NW = kSmallThreads / 32;
    constexpr unsigned long long ROW = (unsigned long long)kSmallThreads * VEC;
    const U ident = Op::template identity<U>();

    __shared__ U s_warp[NW];
    __shared__ U s_carry;
    __shared__ int s_ok;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long n = a.n;
    const T *in = reinterpret_cast<const T *>(a.in);
    T *out = reinterpret_cast<T *>(a.out);

    if (tid == 0) {
        uint32_t epoch;
        s_ok = begin_call(reinterpret_cast<const Header *>(a.ws), &epoch) ? 1 : 0;
        // the only read of carry_in; carry_out is written after every use
        s_carry = a.carry_in ? *reinterpret_cast<const U *>(a.carry_in) : ident;
    }
    // all rows into registers (identity past the end)
    U v[kSmallRows][VEC];
#pragma unroll
    for (int r = 0; r < kSmallRows; ++r) {
        const unsigned long long base = (unsigned long long)r * ROW + (unsigned long long)tid * VEC;
        if (vec_io && base + VEC <= n) {
            const V x = *reinterpret_cast<const V *>(in + base);
#pragma unroll
            for (int j = 0; j < VEC; ++j) v[r][j] = (U)vget(x, j);
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) v[r][j] = base + j < n ? (U)in[base + j] : ident;
        }
    }
    __syncthreads();
    if (!s_ok) return;   // the same in every thread
    U carry = s_carry;

#pragma unroll
    for (int r = 0; r < kSmallRows; ++r) {
        if ((unsigned long long)r * ROW >= n) break;   // the same in every thread
        // this thread's vector, serially
        U t;
        if (EXCL) {
            U acc = ident;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const U x = v[r][j];
                v[r][j] = acc;
                acc = Op::combine(acc, x);
            }
            t = acc;
        } else {
#pragma unroll
            for (int j = 1; j < VEC; ++j) v[r][j] = Op::combine(v[r][j - 1], v[r][j]);
            t = v[r][VEC - 1];
        }
        // the lanes, then the warps
        const U sc = warp_inclusive<U, Op>(t, lane);
        U lane_excl = __shfl_up_sync(kFull, sc, 1);
        if (lane == 0) lane_excl = ident;
        if (lane == 31) s_warp[warp] = sc;
        __syncthreads();
        if (warp == 0) s_warp[lane] = warp_inclusive<U, Op>(s_warp[lane], lane);
        __syncthreads();
        const U warp_excl = warp > 0 ? s_warp[warp - 1] : ident;
        const U row_total = s_warp[NW - 1];
        const U pre = Op::combine(carry, Op::combine(warp_excl, lane_excl));
#pragma unroll
        for (int j = 0; j < VEC; ++j) v[r][j] = Op::combine(pre, v[r][j]);
        carry = Op::combine(carry, row_total);
        __syncthreads();   // s_warp is reused by the next row
    }

#pragma unroll
    for (int r = 0; r < kSmallRows; ++r) {
        const unsigned long long base = (unsigned long long)r * ROW + (unsigned long long)tid * VEC;
        if (vec_io && base + VEC <= n) {
            V w;
#pragma unroll
            for (int j = 0; j < VEC; ++j) vset(w, j, v[r][j]);
            *reinterpret_cast<V *>(out + base) = w;
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (base + j < n) out[base + j] = (T)v[r][j];
        }
    }
    if (tid == 0 && a.carry_out) *reinterpret_cast<U *>(a.carry_out) = carry;
}

template <typename T, typename Op>
static cudaError_t launch_small_op(const PassArgs &a, bool exclusive, cudaStream_t s) {
    const int vec_io = ((reinterpret_cast<uintptr_t>(a.in) | reinterpret_cast<uintptr_t>(a.out)) & 15u) == 0;
    if (exclusive)
        small_scan_kernel<T, true, Op><<<1, kSmallThreads, 0, s>>>(a, vec_io);
    else
        small_scan_kernel<T, false, Op><<<1, kSmallThreads, 0, s>>>(a, vec_io);
    return cudaGetLastError();
}

template <typename T>
unsigned long long small_scan_limit() {
    return small_scan_max<T>();
}

template <typename T>
cudaError_t launch_small(const PassArgs &a, bool exclusive, int op, cudaStream_t s) {
    if constexpr (sizeof(T) == 8) {
        if (op == kOpPairI32F32) return launch_small_op<T, OpPairI32F32>(a, exclusive, s);
        if (op == kOpAffineF32) return launch_small_op<T, OpAffineF32>(a, exclusive, s);
    }
    switch (op) {
    case kOpMax: return launch_small_op<T, OpMax>(a, exclusive, s);
    case kOpMin: return launch_small_op<T, OpMin>(a, exclusive, s);
    default: return launch_small_op<T, OpSum>(a, exclusive, s);
    }
}

template unsigned long long small_scan_limit<int32_t>();
template unsigned long long small_scan_limit<int64_t>();
template unsigned long long small_scan_limit<float>();
template cudaError_t launch_small<int32_t>(const PassArgs &, bool, int, cudaStream_t);
template cudaError_t launch_small<int64_t>(const PassArgs &, bool, int, cudaStream_t);
template cudaError_t launch_small<float>(const PassArgs &, bool, int, cudaStream_t);

}  // namespace ps
