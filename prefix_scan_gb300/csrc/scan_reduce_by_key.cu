// scan_reduce_by_key.cu -- single-pass reduce-by-key (decoupled look-back
// paper summary, A5: one of the fused compaction workloads besides select
// and partition).
//
// Element i opens a run ("head") when i == 0 or its key bits differ from
// those of element i-1.  With the pair p_i = (head_i, value_i) and the
// segmented-sum operator
//     (c1, v1) (+) (c2, v2) = (c1 + c2,  c2 != 0 ? v2 : v1 + v2),
// the inclusive scan at i is (heads up to i, sum of the values of i's run up
// to i).  So a head i with exclusive scan (c, v) starts run c, and v is the
// complete value of run c-1: the scatter writes unique_keys[c] = key_i and
// aggregates[c-1] = v; the inclusive scan at n-1 gives the last run's value
// and the number of runs.  The operator is associative but not commutative;
// the method only ever combines contiguous partials (section 4.2), so the
// look-back works unchanged once its window reduction keeps the order.
// (Run-length encoding needs no value sums -- a run's length is the
// distance between two heads -- and has its own kernel, scan_rle.cu.)
//
// The pair travels as one 64-bit word, count << 32 | value bits, and a tile
// descriptor is the two-word form the int64 scan uses.
//
// Structure as in the persistent scan and the compaction kernels: a producer
// warp takes tile ids and bulk-copies the tile's keys -- starting one
// 16-byte vector early, so the key before the tile (the "halo") is in shared
// memory too -- and values into a 3-stage ring; an aggregator warp computes
// the tile's pair and publishes it at once; a look-back warp resolves the
// tile's exclusive pair; eight compute warps scan the tile and scatter.  The
// aggregator needs no ordered reduction: the count is a plain sum, and the
// value is the sum of the values from the tile's last head on (all of them
// when it has none), found with a maximum.
#include "scan_device.cuh"
#include "scan_pipeline.cuh"
#include "scan_trace.cuh"

namespace ps {

namespace {

constexpr int kRCW = kThreads / 32;   // compute warps per CTA
constexpr int kRStages = 3;
// Aggregator warps per CTA (a macro so that a tuning sweep can rebuild).
#ifndef PS_RBK_AGG_WARPS
#define PS_RBK_AGG_WARPS 4
#endif
constexpr int kAgg = PS_RBK_AGG_WARPS;
// Look-back warps per CTA: each resolves every kLB-th tile of the CTA, so
// that one CTA has several look-backs in flight (a single look-back warp
// caps a CTA at one tile per look-back latency).
#ifndef PS_RBK_LOOKBACK_WARPS
#define PS_RBK_LOOKBACK_WARPS 1
#endif
constexpr int kLB = PS_RBK_LOOKBACK_WARPS;
static_assert(kLB >= 1 && kLB <= kRStages, "at most one look-back warp per stage");
constexpr int kRbkThreads = (kRCW + 1 + kLB + kAgg) * 32;   // compute, producer, look-back, aggregators
// Every barrier wait suspends the warp in the barrier for up to this many
// nanoseconds per try (0: poll), so that waiting warps leave the issue slots
// to the ones that work; a macro so that a tuning sweep can rebuild.
#ifndef PS_RBK_WAIT_NS
#define PS_RBK_WAIT_NS 20000
#endif

// Descriptors each look-back lane inspects per round (window = 32 x this).
#ifndef PS_RBK_LOOKBACK_K
#define PS_RBK_LOOKBACK_K PS_LOOKBACK_K
#endif

// Position of packed entry q in a warp's slice: XOR-swizzled within each 32
// entries (a permutation of the block, so the slice's bounds hold).
__device__ __forceinline__ uint32_t rbk_sw(uint32_t q) { return q ^ ((q >> 5) & 7u); }
__device__ __forceinline__ bool role_wait(uint64_t *bar, uint32_t parity) {
    return PS_RBK_WAIT_NS ? mbar_wait_suspend(bar, parity, PS_RBK_WAIT_NS) : mbar_wait(bar, parity);
}

template <typename VU> struct RunValue;
template <> struct RunValue<uint32_t> {   // int32 values, modulo 2^32
    static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) { return a + b; }
    static __device__ __forceinline__ uint32_t warp_total(uint32_t v) { return __reduce_add_sync(kFull, v); }
};
template <> struct RunValue<float> {      // fp32 values, carried as their bits
    static __device__ __forceinline__ uint32_t add(uint32_t a, uint32_t b) {
        return __float_as_uint(__uint_as_float(a) + __uint_as_float(b));
    }
    static __device__ __forceinline__ uint32_t warp_total(uint32_t v) {
        float f = __uint_as_float(v);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) f += __shfl_xor_sync(kFull, f, d);
        return __float_as_uint(f);
    }
};

__device__ __forceinline__ unsigned long long pair_of(uint32_t c, uint32_t v) {
    return ((unsigned long long)c << 32) | v;
}
__device__ __forceinline__ uint32_t pair_count(unsigned long long p) { return (uint32_t)(p >> 32); }
__device__ __forceinline__ uint32_t pair_value(unsigned long long p) { return (uint32_t)p; }

// The segmented-sum operator on packed pairs; `a` is the earlier part.
template <typename VU> struct OpSeg {
    static constexpr bool kCommutative = false;
    template <typename U> static __device__ __forceinline__ U identity() { return U(0); }
    template <typename U> static __device__ __forceinline__ U combine(U a, U b) {
        const uint32_t cb = pair_count(b);
        const uint32_t v = cb ? pair_value(b) : RunValue<VU>::add(pair_value(a), pair_value(b));
        return pair_of(pair_count(a) + cb, v);
    }
};

// 16-byte key vectors: four 32-bit keys or two 64-bit keys; the values of
// the same elements, four or two 32-bit words.
template <typename KU> struct KeyVec;
template <> struct KeyVec<uint32_t> {
    using V = uint4;
    using W = uint4;   // the values of the same four elements
    static constexpr int N = 4;
    static __device__ __forceinline__ uint32_t key(const V &v, int j) { return vget(v, j); }
    static __device__ __forceinline__ uint32_t val(const W &w, int j) { return vget(w, j); }
};
template <> struct KeyVec<unsigned long long> {
    using V = ulonglong2;
    using W = uint2;
    static constexpr int N = 2;
    static __device__ __forceinline__ unsigned long long key(const V &v, int j) { return vget(v, j); }
    static __device__ __forceinline__ uint32_t val(const W &w, int j) { return j == 0 ? w.x : w.y; }
};

// Keys per tile for 32-bit keys (half as many for 64-bit ones); a macro so
// that a tuning sweep can rebuild (the workspace is sized for 4096).
#ifndef PS_RBK_TILE32
#define PS_RBK_TILE32 4096
#endif
template <typename KU> constexpr long long rbk_tile() { return sizeof(KU) == 4 ? PS_RBK_TILE32 : PS_RBK_TILE32 / 2; }
template <typename KU> constexpr uint32_t rbk_key_bytes() {   // the tile's keys and the halo vector
    return (uint32_t)(rbk_tile<KU>() * sizeof(KU) + 16);
}
template <typename KU> constexpr uint32_t rbk_stage_bytes() {
    return rbk_key_bytes<KU>() + (uint32_t)(rbk_tile<KU>() * 4);
}
template <typename KU> constexpr size_t rbk_smem_bytes() {
    return (size_t)kRStages * rbk_stage_bytes<KU>() + ((size_t)kRStages * (4 * 8 + 8 * 3) + 8 + 127) / 128 * 128;
}

}  // namespace


template <typename KU, typename VU>
__global__ void __launch_bounds__(kRbkThreads, kPCtasPerSm)
reduce_by_key_kernel(RbkArgs a, long long num_tiles) {
    using KV = KeyVec<KU>;
    using V = typename KV::V;
    using W = typename KV::W;
    using Op = OpSeg<VU>;
    using P = unsigned long long;
    constexpr int VK = KV::N;
    constexpr long long TILE = rbk_tile<KU>();
    constexpr int ITEMS = (int)(TILE / kThreads);
    // A compute lane's share of a row: two key vectors (EPL keys) and their
    // EPL 32-bit values (one or two 16-byte vectors), so that a tile takes
    // half as many segmented warp scans as with one key vector per row.
    constexpr int EPL = 2 * VK;
    constexpr int ROWS = ITEMS / EPL;
    constexpr int WV = EPL / 4;   // 16-byte value vectors per lane per row
    constexpr int S = kRStages;
    constexpr uint32_t KEY_BYTES = rbk_key_bytes<KU>();
    constexpr uint32_t STAGE = rbk_stage_bytes<KU>();
    constexpr uint32_t VAL_BYTES = (uint32_t)(TILE * 4);
    constexpr int CT = kRCW * 32;
    static_assert(ITEMS % EPL == 0 && (WV == 1 || WV == 2) && STAGE % 16 == 0, "tile geometry");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * STAGE);
    uint64_t *empty = full + S;
    uint64_t *agg_done = empty + S;
    uint64_t *prefix_ready = agg_done + S;
    uint64_t *agg_bar = prefix_ready + S;   // the aggregator warps meet here (bounded waits)
    long long *tile_of = reinterpret_cast<long long *>(agg_bar + 1);
    P *agg_of = reinterpret_cast<P *>(tile_of + S);
    P *excl_of = agg_of + S;
    __shared__ P s_warp[2][kRCW];
    __shared__ int s_abort;   // a compute warp's wait ran out: all of them leave
    __shared__ uint32_t s_ah[2][kAgg], s_av[2][kAgg];   // aggregator shares: heads, values
    __shared__ int s_al[2][kAgg];                       // and last head
    // stage s: [halo vector][TILE keys][TILE values]
    auto stage_keys = [&](int s) { return reinterpret_cast<KU *>(smem + (size_t)s * STAGE) + VK; };
    auto stage_vals = [&](int s) { return reinterpret_cast<uint32_t *>(smem + (size_t)s * STAGE + KEY_BYTES); };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Header *hdr = reinterpret_cast<Header *>(a.ws);
    void *desc = a.ws + kHeaderBytes;
    const unsigned long long n = a.n;
    const KU *keys = reinterpret_cast<const KU *>(a.keys);
    const uint32_t *vals = reinterpret_cast<const uint32_t *>(a.vals);
    KU *ukeys = reinterpret_cast<KU *>(a.unique_keys);
    uint32_t *aggs = reinterpret_cast<uint32_t *>(a.aggs);

    // thread 0 alone reads the header (one request per CTA to its line)
    __shared__ uint32_t s_epoch;
    __shared__ int s_ok;
    if (tid == 0) {
        PS_TRACE_CTA_POINT(PS_TRACE_CTA_ENTRY);
        if (PS_PREFETCH_FIRST_TILES && a.use_bulk) {
            for (int j = 0; j < S; ++j) {
                const unsigned long long t = blockIdx.x + (unsigned long long)j * gridDim.x;
                if ((t + 1) * (unsigned long long)TILE <= n) {
                    prefetch_l2(keys + t * TILE, (uint32_t)(TILE * sizeof(KU)));   // the tile, no halo
                    prefetch_l2(vals + t * TILE, VAL_BYTES);
                }
            }
        }
        uint32_t e;
        s_ok = begin_call(hdr, &e) ? 1 : 0;
        s_epoch = e;
        s_abort = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRCW + kAgg);
            mbar_init(&agg_done[s], 1);
            mbar_init(&prefix_ready[s], 1);
            tile_of[s] = num_tiles;
        }
        mbar_init(agg_bar, kAgg);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!s_ok) return;   // same verdict in every CTA
    const uint32_t epoch = s_epoch;
    if (tid == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_HEADER);

    if (warp == kRCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int ends = 0;   // end markers sent: one per look-back warp
            for (long long k = 0;; ++k) {
                const int s = (int)(k % S);
                if (k >= S && !role_wait(&empty[s], (uint32_t)((k / S - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    break;
                }
                const long long t = ends ? num_tiles : (long long)atomicAdd(&hdr->tile_counter, 1ull);
                tile_of[s] = t;
                if (t < num_tiles) {
                    prefetch_descriptor<2>(desc, t);
                    PS_TRACE_POINT(t, PS_TRACE_CLAIM);
                    PS_TRACE_CTA(t);
                }
                if (a.use_bulk && t < num_tiles && (unsigned long long)(t + 1) * TILE <= n) {
                    const uint32_t kb = t == 0 ? KEY_BYTES - 16u : KEY_BYTES;
                    mbar_arrive_expect_tx(&full[s], kb + VAL_BYTES);
                    if (t == 0)
                        bulk_load(stage_keys(s), keys, kb, &full[s]);
                    else
                        bulk_load(stage_keys(s) - VK, keys + t * TILE - VK, kb, &full[s]);
                    bulk_load(stage_vals(s), vals + t * TILE, VAL_BYTES, &full[s]);
                } else {
                    mbar_arrive(&full[s]);   // end marker, or a tile read from global
                }
                if (t >= num_tiles && ++ends == kLB) break;
            }
            if (epoch != kEpochMask) claims_done(hdr, a.ws_bytes, epoch);
        }
    } else if (warp > kRCW && warp <= kRCW + kLB) {
        // ---------------- look-back warps: the tile's exclusive pair ----------------
        for (long long k = warp - (kRCW + 1);; k += kLB) {
            const int s = (int)(k % S);
            if (!role_wait(&agg_done[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[s];
            if (tile < 0 || tile >= num_tiles) break;
            const P agg = agg_of[s];
            if (lane == 0) PS_TRACE_POINT(tile, PS_TRACE_LOOKBACK_START);
            __syncwarp();
            P excl = 0;
            if (tile != 0) {
                excl = look_back<P, 2, PS_RBK_LOOKBACK_K, Op>(desc, tile, epoch, a.max_polls, &hdr->status,
                                                              PS_TRACE_LOOKBACK(tile));
                if (lane == 0) Desc<P, 2>::store(desc, tile, kFlagP, Op::combine(excl, agg), epoch);
            }
            if (lane == 0) {
                if (tile == num_tiles - 1) {
                    // the inclusive pair at n-1: number of runs, value of the last one
                    const P incl = Op::combine(excl, agg);
                    const uint32_t runs = pair_count(incl);
                    if (runs > 0) aggs[runs - 1] = pair_value(incl);
                    if (a.num_runs) *a.num_runs = runs;
                }
                excl_of[s] = excl;
                PS_TRACE_POINT(tile, PS_TRACE_PREFIX);
                mbar_arrive(&prefix_ready[s]);
            }
        }
    } else if (warp > kRCW + kLB) {
        // ---------------- aggregators: the tile's pair, published at once ----------------
        // kAgg warps, each over its share of the tile: count the heads and
        // find the last one, combine through shared memory, then sum the
        // values from the tile's last head on, again in shares.
        const int ag = warp - (kRCW + 1 + kLB);
        int ends = 0;   // end markers passed on: one per look-back warp
        constexpr int PART = (int)(TILE / VK / kAgg);   // vectors per aggregator warp
        static_assert(PART % 32 == 0, "aggregator shares must be whole warp rows");
        uint32_t meets = 0;   // completed phases of agg_bar
        auto meet = [&]() {   // all aggregator warps here; false if the wait ran out
            __syncwarp();
            if (lane == 0) mbar_arrive(agg_bar);
            const bool ok = role_wait(agg_bar, meets & 1u);
            ++meets;
            if (!ok) report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
            return ok;
        };
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!role_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[s];
            if (tile < 0 || tile >= num_tiles) {
                if (ag == 0 && lane == 0) mbar_arrive(&agg_done[s]);
                if (++ends == kLB) break;
                continue;
            }
            if (ag == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_DATA);
            const unsigned long long base = (unsigned long long)tile * TILE;
            const bool staged = a.use_bulk && base + TILE <= n;
            const int len = staged ? (int)TILE : (int)(n - base < (unsigned long long)TILE ? n - base : TILE);
            const KU *ks = stage_keys(s);
            uint32_t heads = 0;
            int last = -1;   // tile-local index of the last head in this warp's share
            if (staged) {
                const V *kv = reinterpret_cast<const V *>(ks);
                // the key before the share: the halo (or, for tile 0, a value
                // that differs from element 0, which opens a run), or the
                // previous share's last key
                const KU before = ag > 0 ? ks[ag * PART * VK - 1] : tile == 0 ? (KU)~ks[0] : ks[-1];
                int last_vec = -1;
#pragma unroll 4
                for (int it = 0; it < PART / 32; ++it) {
                    const int vi = ag * PART + it * 32 + lane;
                    const V x = kv[vi];
                    KU prev = __shfl_up_sync(kFull, KV::key(x, VK - 1), 1);
                    if (lane == 0) prev = it == 0 ? before : ks[vi * VK - 1];
                    uint32_t h = 0;
#pragma unroll
                    for (int j = 0; j < VK; ++j) h += (uint32_t)(KV::key(x, j) != (j ? KV::key(x, j - 1) : prev));
                    heads += h;
                    last_vec = h ? vi : last_vec;
                }
                const int lv = __reduce_max_sync(kFull, last_vec);
                if (lv >= 0) {   // the last head within that vector (same in every lane)
                    const V x = kv[lv];
                    const KU prev = lv == ag * PART ? before : ks[lv * VK - 1];
                    uint32_t m = 0;
#pragma unroll
                    for (int j = 0; j < VK; ++j) m |= (uint32_t)(KV::key(x, j) != (j ? KV::key(x, j - 1) : prev)) << j;
                    last = lv * VK + 31 - __clz(m);
                }
            } else if (ag == 0) {   // a tile read from global memory: the first warp alone
                for (int e = lane; e < len; e += 32) {
                    const unsigned long long i = base + e;
                    if (i == 0 || keys[i] != keys[i - 1]) { ++heads; last = e; }
                }
            }
            heads = __reduce_add_sync(kFull, heads);
            last = __reduce_max_sync(kFull, last);
            const int b = (int)(k & 1);
            if (lane == 0) { s_ah[b][ag] = heads; s_al[b][ag] = last; }
            if (!meet()) break;
            uint32_t C = 0;
            int L = -1;
#pragma unroll
            for (int g = 0; g < kAgg; ++g) { C += s_ah[b][g]; L = s_al[b][g] > L ? s_al[b][g] : L; }
            const int from = L < 0 ? 0 : L;   // the tile's trailing run starts here
            uint32_t val = 0u;   // +0.0f for fp32
            uint32_t acc = 0u;
            if (staged) {
                const W *wv = reinterpret_cast<const W *>(stage_vals(s));
                const int v0 = ag * PART, v1 = v0 + PART;
                for (int vi = (from / VK > v0 ? from / VK : v0) + lane; vi < v1; vi += 32) {
                    const W w = wv[vi];
#pragma unroll
                    for (int j = 0; j < VK; ++j)
                        if (vi * VK + j >= from) acc = RunValue<VU>::add(acc, KV::val(w, j));
                }
            } else if (ag == 0) {
                for (int e = from + lane; e < len; e += 32) acc = RunValue<VU>::add(acc, vals[base + e]);
            }
            acc = RunValue<VU>::warp_total(acc);
            if (lane == 0) s_av[b][ag] = acc;
            if (!meet()) break;
#pragma unroll
            for (int g = 0; g < kAgg; ++g) val = RunValue<VU>::add(val, s_av[b][g]);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s]);
                if (ag == 0) {
                    const P agg = pair_of(C, val);
                    Desc<P, 2>::store(desc, tile, tile == 0 ? kFlagP : kFlagA, agg, epoch);
                    PS_TRACE_POINT(tile, PS_TRACE_AGGREGATE);
                    agg_of[s] = agg;
                    mbar_arrive(&agg_done[s]);
                }
            }
        }
    } else {
        // ---------------- compute warps: scan the pairs, scatter at heads ----------------
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!role_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                abort_meet(&s_abort, 1, CT);
                break;
            }
            const long long tile = tile_of[s];
            if (tile < 0 || tile >= num_tiles) break;
            const unsigned long long base = (unsigned long long)tile * TILE;
            const bool staged = a.use_bulk && base + TILE <= n;
            const int seg = warp * 32 * ITEMS;
            if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_COMPUTE_START);

            KU kk[ROWS][EPL];
            uint32_t vv[ROWS][EPL];
            uint32_t hm[ROWS];              // bit j: element j of this lane's chunk opens a run
            uint32_t offc[ROWS], offv[ROWS];   // exclusive pair of the chunk within the warp
            uint32_t rc = 0u, rv = 0u;      // pair of the warp's rows so far
            const uint32_t lt_mask = (1u << lane) - 1u;
            // lanes 4-7 of each quarter-warp read a pair of 16-byte vectors
            // in swapped order, so that the quarter-warp's reads fall in
            // distinct bank groups; the pair is put back in order in registers
            const int rot = (lane >> 2) & 1;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int e0 = seg + (r * 32 + lane) * EPL;   // tile-local index of the chunk
                uint32_t m = 0;
                if (staged) {
                    const KU *ks = stage_keys(s);
                    const V *kv = reinterpret_cast<const V *>(ks) + e0 / VK;
                    const V x0 = kv[rot], x1 = kv[rot ^ 1];
                    const V klo = rot ? x1 : x0, khi = rot ? x0 : x1;
#pragma unroll
                    for (int j = 0; j < VK; ++j) {
                        kk[r][j] = KV::key(klo, j);
                        kk[r][VK + j] = KV::key(khi, j);
                    }
                    KU prev = __shfl_up_sync(kFull, kk[r][EPL - 1], 1);
                    if (lane == 0) prev = ks[e0 - 1];   // e0 == 0 reads the halo
#pragma unroll
                    for (int j = 0; j < EPL; ++j) m |= (uint32_t)(kk[r][j] != (j ? kk[r][j - 1] : prev)) << j;
                    if (tile == 0 && e0 == 0) m |= 1u;
                    const uint4 *wv = reinterpret_cast<const uint4 *>(stage_vals(s)) + e0 / 4;
                    if constexpr (WV == 2) {
                        const uint4 w0 = wv[rot], w1 = wv[rot ^ 1];
                        const uint4 vlo = rot ? w1 : w0, vhi = rot ? w0 : w1;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            vv[r][j] = vget(vlo, j);
                            vv[r][4 + j] = vget(vhi, j);
                        }
                    } else {
                        const uint4 w = wv[0];
#pragma unroll
                        for (int j = 0; j < 4; ++j) vv[r][j] = vget(w, j);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < EPL; ++j) {
                        const unsigned long long i = base + (unsigned long long)(e0 + j);
                        if (i < n) {
                            kk[r][j] = keys[i];
                            m |= (uint32_t)(i == 0 || kk[r][j] != keys[i - 1]) << j;
                            vv[r][j] = vals[i];
                        } else {
                            kk[r][j] = KU(0);
                            vv[r][j] = 0u;   // past the end: neither a head nor a value
                        }
                    }
                }
                hm[r] = m;
            }
            // Segmented inclusive scan of the chunk pairs over the lanes, the
            // rows side by side so that their shuffle chains overlap.  A
            // chunk's pair is (its heads, its value from its last head on);
            // the segment of lane l starts at the nearest lane <= l whose
            // chunk holds a head (none: it reaches back past lane 0), and a
            // partial from lane l-d joins only while l-d lies in it.
            uint32_t cc[ROWS], cv[ROWS], cnt[ROWS];
            int seg_lo[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                uint32_t v = 0u;
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const bool h = (hm[r] >> j) & 1u;
                    const uint32_t sum = RunValue<VU>::add(v, vv[r][j]);
                    v = h ? vv[r][j] : sum;
                }
                cv[r] = v;
                cnt[r] = (uint32_t)__popc(hm[r]);
                cc[r] = cnt[r];
                const uint32_t with_head = __ballot_sync(kFull, hm[r] != 0u);
                const uint32_t le = with_head & (lt_mask | (1u << lane));
                seg_lo[r] = le ? 31 - __clz(le) : -1;
            }
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint32_t oc = __shfl_up_sync(kFull, cc[r], d);
                    const uint32_t ov = __shfl_up_sync(kFull, cv[r], d);
                    const uint32_t sum = RunValue<VU>::add(ov, cv[r]);
                    cc[r] += lane >= d ? oc : 0u;
                    cv[r] = (lane >= d && lane - d >= seg_lo[r]) ? sum : cv[r];
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                // exclusive pair of the chunk: lane l-1's inclusive pair
                const uint32_t ec = cc[r] - cnt[r];
                uint32_t ev = __shfl_up_sync(kFull, cv[r], 1);
                if (lane == 0) ev = 0u;
                offc[r] = rc + ec;
                offv[r] = ec ? ev : RunValue<VU>::add(rv, ev);
                const uint32_t tc = __shfl_sync(kFull, cc[r], 31), tv = __shfl_sync(kFull, cv[r], 31);
                rv = tc ? tv : RunValue<VU>::add(rv, tv);
                rc += tc;
            }
            P *sw = s_warp[k & 1];
            if (lane == 0) sw[warp] = pair_of(rc, rv);
            named_barrier(1, CT);
            if (aborted(&s_abort)) break;
            P warp_excl = 0;
#pragma unroll
            for (int w = 0; w < kRCW; ++w)
                if (w < warp) warp_excl = Op::combine(warp_excl, sw[w]);
            if (!role_wait(&prefix_ready[s], (uint32_t)((k / S) & 1)))
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
            const P pre = Op::combine(excl_of[s], warp_excl);
            if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_PREFIX_RECEIVED);
            // Pack this warp's runs in its own slice of the stage -- free now:
            // every compute warp has read the stage (named barrier above) and
            // the aggregator finished with it before the prefix was handed
            // over -- keyed by run index relative to the warp's first run,
            // then write them out as two contiguous ranges: keys of runs
            // cw .. cw+rc-1 and values of runs cw-1 .. cw+rc-2 (each head
            // closes the run before it).  Entries are XOR-swizzled within
            // each 32 (rbk_sw), so lanes packing entries EPL apart (every key
            // a head) and lanes reading 32 consecutive ones hit distinct banks.
            const uint32_t cw = pair_count(pre), pv = pair_value(pre);
            KU *pk = stage_keys(s) + seg;
            uint32_t *pvals = stage_vals(s) + seg;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                uint32_t q = offc[r];   // run index - cw of this chunk's first head
                uint32_t v = offc[r] ? offv[r] : RunValue<VU>::add(pv, offv[r]);
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const bool h = (hm[r] >> j) & 1u;
                    if (h) {
                        pk[rbk_sw(q)] = kk[r][j];
                        pvals[rbk_sw(q)] = v;
                    }
                    const uint32_t sum = RunValue<VU>::add(v, vv[r][j]);
                    v = h ? vv[r][j] : sum;
                    q += h ? 1u : 0u;
                }
            }
            __syncwarp();
            for (uint32_t q = lane; q < rc; q += 32) {
                ukeys[cw + q] = pk[rbk_sw(q)];
                if (cw + q > 0u) aggs[cw + q - 1u] = pvals[rbk_sw(q)];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_STORED);
        }
        if (warp == 0 && lane == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_DONE);
    }

    // the last producer readied the workspace; before an epoch wrap the
    // last CTA to finish does
    if (epoch == kEpochMask) finish_call(hdr, a.ws, a.ws_bytes, epoch);
}

template <typename KU, typename VU>
static cudaError_t launch_rbk_variant(const RbkArgs &a, cudaStream_t s) {
    constexpr size_t smem = rbk_smem_bytes<KU>();
    const long long tiles = (long long)((a.n + rbk_tile<KU>() - 1) / rbk_tile<KU>());
    static volatile int configured[64] = {};
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(reduce_by_key_kernel<KU, VU>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    long long grid = (long long)sms * kPCtasPerSm;
    if (grid > tiles) grid = tiles;
    reduce_by_key_kernel<KU, VU><<<(unsigned int)grid, kRbkThreads, smem, s>>>(a, tiles);
    return cudaGetLastError();
}

template <typename KU>
static cudaError_t launch_rbk_keys(const RbkArgs &a, ps_dtype val_dt, cudaStream_t s) {
    if (val_dt == PS_FLOAT32) return launch_rbk_variant<KU, float>(a, s);
    return launch_rbk_variant<KU, uint32_t>(a, s);
}

cudaError_t launch_reduce_by_key(const RbkArgs &a, ps_dtype key_dt, ps_dtype val_dt, cudaStream_t s) {
    static_assert(rbk_tile<uint32_t>() >= (long long)rbk_tile_elems(PS_INT32) &&
                  rbk_tile<unsigned long long>() >= (long long)rbk_tile_elems(PS_INT64),
                  "the workspace must hold a descriptor per tile of the kernel");
    return key_dt == PS_INT64 ? launch_rbk_keys<unsigned long long>(a, val_dt, s)
                              : launch_rbk_keys<uint32_t>(a, val_dt, s);
}

TRACE_COPY_FUNCTIONS(trace_copy_rbk, trace_copy_rbk_ctas)

}  // namespace ps
