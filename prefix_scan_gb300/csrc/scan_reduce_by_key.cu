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
// Roles (as in scan_rle.cu).  A producer warp takes tile ids and bulk-copies
// each tile's keys -- starting one 16-byte vector early, so the key before
// the tile (the "halo") is in shared memory too -- and values into a ring
// of stages.  Eight compute warps take the tiles in order and never wait
// for a tile's prefix: they scan the tile's pairs (a segmented shuffle scan
// of all rows side by side), combine the warps' pairs into the tile's pair
// and publish it (A; P for tile 0) themselves, and pack the tile's runs in
// order into an output buffer -- each head's key and the value of the run it
// closes, summed within the tile -- after which the stage goes back to the
// producer.  The walk over each lane's chunk that precedes the scan leaves
// each head's closing value in the warp's slice of the stage, so the pack
// visits the heads only.  Only the run closed by the tile's first head
// reaches back before the tile; its packed value lacks the value the tile's
// exclusive pair carries.  Look-back warps resolve that pair; a writer warp
// adds its value to the first run and writes the buffer out as contiguous
// ranges, then frees the buffer.  A tile with more runs than a buffer holds
// (a dense tile) is written by the compute warps themselves, one iteration
// late: they publish its pair, keep its stage, do the next tile's pass (so
// that tile's pair is out too), then wait for the dense tile's prefix,
// re-read its keys and the closing values, and pack and write each warp's
// runs from its slice of the stage.
#include "scan_device.cuh"
#include "scan_pipeline.cuh"
#include "scan_trace.cuh"

namespace ps {

namespace {

// Compute warps per CTA and CTAs per SM (macros, so that a tuning sweep can
// rebuild).
#ifndef PS_RBK_COMPUTE_WARPS
#define PS_RBK_COMPUTE_WARPS 8
#endif
#ifndef PS_RBK_CTAS_PER_SM
#define PS_RBK_CTAS_PER_SM 2
#endif
constexpr int kRCW = PS_RBK_COMPUTE_WARPS;
constexpr int kRCtasPerSm = PS_RBK_CTAS_PER_SM;
static_assert(kRCW >= 1 && kRCW <= 32, "the warps' pairs are scanned across the lanes of one warp");
// Stages, output buffers and their bytes, look-back and writer warps (macros
// so that a tuning sweep can rebuild).
#ifndef PS_RBK_STAGES
#define PS_RBK_STAGES 3
#endif
#ifndef PS_RBK_OUT_BUFFERS
#define PS_RBK_OUT_BUFFERS 4
#endif
#ifndef PS_RBK_OUT_BYTES
#define PS_RBK_OUT_BYTES 4096
#endif
#ifndef PS_RBK_LOOKBACK_WARPS
#define PS_RBK_LOOKBACK_WARPS 2
#endif
#ifndef PS_RBK_WRITER_WARPS
#define PS_RBK_WRITER_WARPS 1
#endif
constexpr int kRStages = PS_RBK_STAGES;
constexpr int kROut = PS_RBK_OUT_BUFFERS;
constexpr int kROutBytes = PS_RBK_OUT_BYTES;
constexpr int kLB = PS_RBK_LOOKBACK_WARPS;
constexpr int kRW = PS_RBK_WRITER_WARPS;
constexpr int rmax(int a, int b) { return a > b ? a : b; }
// Iterations past the end the compute warps mark (every look-back and
// writer warp waits on its next iteration), and the hand-off slots: a slot
// is reused only after every role is done with it -- the writer is at most
// kROut iterations behind the compute warps, the producer at most
// kRStages + 1 ahead of their pass.
constexpr int kREnds = rmax(kLB, kRW);
constexpr int rbk_ring_slots() { return (rmax(kRStages + kROut + 1, kREnds + kROut) + 1) / 2 * 2; }
constexpr int kRRing = rbk_ring_slots();
constexpr int kRbkThreads = (kRCW + 1 + kLB + kRW) * 32;   // compute, producer, look-back, writer
static_assert(kRStages >= 2, "a dense tile keeps its stage while the next one is scanned");
// Barrier waits poll (0), or suspend the warp in the barrier for up to this
// many nanoseconds per try; a macro so that a tuning sweep can rebuild.
// Polling measured 3-4 % faster than 20 us suspends (2^28, mean run 16:
// 477.7 -> 462.5 us), where waking from the suspend comes late.
#ifndef PS_RBK_WAIT_NS
#define PS_RBK_WAIT_NS 0
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
// Runs an output buffer holds: a key and a 32-bit value each, a multiple of
// 32 entries (the swizzle stays within each 32).
template <typename KU> constexpr int rbk_out_cap() { return (int)((kROutBytes / (sizeof(KU) + 4)) / 32 * 32); }
template <typename KU> constexpr size_t rbk_smem_bytes() {
    return (size_t)kRStages * rbk_stage_bytes<KU>() + (size_t)kROut * kROutBytes +
           ((size_t)kRStages * 2 * 8 + (size_t)kROut * 8 + (size_t)kRRing * (3 * 8 + 4 * 8) + 127) / 128 * 128;
}

}  // namespace


template <typename KU, typename VU>
__global__ void __launch_bounds__(kRbkThreads, kRCtasPerSm)
reduce_by_key_kernel(RbkArgs a, long long num_tiles) {
    using KV = KeyVec<KU>;
    using V = typename KV::V;
    using Op = OpSeg<VU>;
    using P = unsigned long long;
    constexpr int VK = KV::N;
    constexpr long long TILE = rbk_tile<KU>();
    constexpr int ITEMS = (int)(TILE / (kRCW * 32));
    // A compute lane's share of a row: two key vectors (EPL keys) and their
    // EPL 32-bit values (one or two 16-byte vectors), so that a tile takes
    // half as many segmented warp scans as with one key vector per row.
    constexpr int EPL = 2 * VK;
    constexpr int ROWS = ITEMS / EPL;
    constexpr int WV = EPL / 4;   // 16-byte value vectors per lane per row
    constexpr int S = kRStages, R = kRRing, NOB = kROut;
    constexpr uint32_t KEY_BYTES = rbk_key_bytes<KU>();
    constexpr uint32_t STAGE = rbk_stage_bytes<KU>();
    constexpr uint32_t VAL_BYTES = (uint32_t)(TILE * 4);
    constexpr int CT = kRCW * 32;
    constexpr int CAP = rbk_out_cap<KU>();
    static_assert(ITEMS % EPL == 0 && (WV == 1 || WV == 2) && STAGE % 16 == 0, "tile geometry");
    static_assert(CAP >= 32 && 32 * ITEMS < (1 << 23), "output buffer geometry, packed row words");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *outbuf = smem + (size_t)S * STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(outbuf + (size_t)NOB * kROutBytes);
    uint64_t *empty = full + S;
    uint64_t *ob_empty = empty + S;
    uint64_t *agg_done = ob_empty + NOB;   // the rest: R slots, slot k % R
    uint64_t *prefix_ready = agg_done + R;
    uint64_t *packed = prefix_ready + R;
    long long *tile_of = reinterpret_cast<long long *>(packed + R);
    P *agg_of = reinterpret_cast<P *>(tile_of + R);
    P *excl_of = agg_of + R;
    int *sparse_of = reinterpret_cast<int *>(excl_of + R);
    __shared__ P s_warp[2][kRCW];
    __shared__ int s_abort;   // a compute warp's wait ran out: all of them leave
    // stage s: [halo vector][TILE keys][TILE values]
    auto stage_keys = [&](int s) { return reinterpret_cast<KU *>(smem + (size_t)s * STAGE) + VK; };
    auto stage_vals = [&](int s) { return reinterpret_cast<uint32_t *>(smem + (size_t)s * STAGE + KEY_BYTES); };
    // output buffer o: a sparse tile's runs, CAP keys then CAP values, entry
    // q at rbk_sw(q)
    auto out_keys = [&](int o) { return reinterpret_cast<KU *>(outbuf + (size_t)o * kROutBytes); };
    auto out_vals = [&](int o) {
        return reinterpret_cast<uint32_t *>(outbuf + (size_t)o * kROutBytes + (size_t)CAP * sizeof(KU));
    };

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
        uint32_t e;
        s_ok = begin_call(hdr, &e) ? 1 : 0;
        s_epoch = e;
        s_abort = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRCW);   // each compute warp, once it needs the stage no more
        }
        for (int o = 0; o < NOB; ++o) mbar_init(&ob_empty[o], 1);   // the writer
        for (int slot = 0; slot < R; ++slot) {
            mbar_init(&agg_done[slot], 1);
            mbar_init(&prefix_ready[slot], 1);
            mbar_init(&packed[slot], kRCW);
            tile_of[slot] = num_tiles;   // end marker until the producer fills it
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!s_ok) return;   // same verdict in every CTA
    const uint32_t epoch = s_epoch;
    if (tid == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_HEADER);

    if (warp == kRCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            for (long long k = 0;; ++k) {
                const int s = (int)(k % S);
                if (k >= S && !role_wait(&empty[s], (uint32_t)((k / S - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    break;
                }
                const long long t = (long long)atomicAdd(&hdr->tile_counter, 1ull);
                tile_of[k % R] = t;
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
                if (t >= num_tiles) break;   // the compute warps pass the end marker on
            }
            if (epoch != kEpochMask) claims_done(hdr, a.ws_bytes, epoch);
        }
    } else if (warp > kRCW && warp <= kRCW + kLB) {
        // ---------------- look-back warps: the tile's exclusive pair ----------------
        for (long long k = warp - (kRCW + 1);; k += kLB) {
            const int slot = (int)(k % R);
            if (!role_wait(&agg_done[slot], (uint32_t)((k / R) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            const P agg = agg_of[slot];
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
                excl_of[slot] = excl;
                PS_TRACE_POINT(tile, PS_TRACE_PREFIX);
                mbar_arrive(&prefix_ready[slot]);
            }
        }
    } else if (warp > kRCW + kLB) {
        // ---------------- writer warps: a tile's runs, once its pair is known ----------------
        for (long long k = warp - (kRCW + 1 + kLB);; k += kRW) {
            const int slot = (int)(k % R);
            const uint32_t par = (uint32_t)((k / R) & 1);
            if (!role_wait(&packed[slot], par)) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            if (!role_wait(&prefix_ready[slot], par)) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const int o = (int)(k % NOB);
            const bool sparse = sparse_of[slot] != 0;
            if (sparse) {
                // the runs in order: keys to unique_keys[c0 + t], and the value
                // of the run each head closes to aggregates[c0 + t - 1]; the
                // first of them began before the tile, so the exclusive pair's
                // value (that run's sum so far) is added to its packed part
                if (lane == 0) PS_TRACE_POINT(tile, PS_TRACE_PREFIX_RECEIVED);
                const P excl = excl_of[slot];
                const uint32_t c0 = pair_count(excl), pv = pair_value(excl);
                const uint32_t h = pair_count(agg_of[slot]);
                const KU *ok = out_keys(o);
                const uint32_t *ov = out_vals(o);
                for (uint32_t t = lane; t < h; t += 32) {
                    ukeys[c0 + t] = ok[rbk_sw(t)];
                    if (c0 + t > 0u) aggs[c0 + t - 1u] = t ? ov[rbk_sw(t)] : RunValue<VU>::add(pv, ov[rbk_sw(t)]);
                }
            }   // a dense tile: the compute warps write it
            __syncwarp();
            if (lane == 0) {
                if (sparse) PS_TRACE_POINT(tile, PS_TRACE_STORED);
                mbar_arrive(&ob_empty[o]);
            }
        }
    } else {
        // ---------------- compute warps: scan the pairs, pack the runs ----------------
        const int seg = warp * 32 * ITEMS;   // the warp's first element in a tile
        const uint32_t lt_mask = (1u << lane) - 1u;
        // lanes 4-7 of each quarter-warp read a pair of 16-byte vectors in
        // swapped order, so that the quarter-warp's reads fall in distinct
        // bank groups; the pair is put back in order in registers
        const int rot = (lane >> 2) & 1;
        // This warp's keys and values of a tile, and each lane-chunk's head
        // mask (bit j: element j of the chunk opens a run).
        auto load_rows = [&](int s_, long long tile_, unsigned long long base_, bool staged_, KU (&kk)[ROWS][EPL],
                             uint32_t (&vv)[ROWS][EPL], uint32_t (&hm)[ROWS]) {
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int e0 = seg + (r * 32 + lane) * EPL;   // tile-local index of the chunk
                uint32_t m = 0;
                if (staged_) {
                    const KU *ks = stage_keys(s_);
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
                    if (tile_ == 0 && e0 == 0) m |= 1u;
                    const uint4 *wv = reinterpret_cast<const uint4 *>(stage_vals(s_)) + e0 / 4;
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
                        const unsigned long long i = base_ + (unsigned long long)(e0 + j);
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
        };
        // A dense tile waiting for the next iteration's pass: its stage, slot
        // and the slot's phase parity (stage | slot << 8 | parity << 16), its
        // tile (tile ids of a call with 32-bit run counts fit 32 bits), the
        // pair of its elements before this warp's, this warp's runs, and per
        // row the lane-chunk's head mask (bits 0-7) and runs before it in the
        // warp (bits 8 up), and its exclusive value within the warp.
        bool pend = false;
        uint32_t pend_at = 0, pend_tile = 0, pend_rc = 0;
        P pend_wex = 0;
        uint32_t pend_info[ROWS], pend_offv[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) pend_info[r] = pend_offv[r] = 0;
        // Writes the pending dense tile once its pair is known: this warp's
        // runs packed in its slice of the stage -- keys of runs cw .. cw+rc-1
        // and values of runs cw-1 .. cw+rc-2 (each head closes the run before
        // it) -- then written as two contiguous ranges; the stage goes back
        // after.  Entries are XOR-swizzled within each 32 (rbk_sw), so lanes
        // packing entries EPL apart and lanes reading 32 consecutive ones hit
        // distinct banks.
        auto write_dense = [&]() {
            const int ps = (int)(pend_at & 0xffu), pslot = (int)((pend_at >> 8) & 0xffu);
            const unsigned long long pbase = (unsigned long long)pend_tile * TILE;
            const bool pstaged = a.use_bulk && pbase + TILE <= n;
            if (!role_wait(&prefix_ready[pslot], pend_at >> 16))
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
            if (warp == 0 && lane == 0) PS_TRACE_POINT(pend_tile, PS_TRACE_PREFIX_RECEIVED);
            const P pre = Op::combine(excl_of[pslot], pend_wex);
            const uint32_t cw = pair_count(pre), pv = pair_value(pre);
            // the warp's keys again, and the closing values its pass left in
            // the slice, all of them before the slice is reused (the values
            // loaded beside the keys are not used)
            KU kp[ROWS][EPL];
            uint32_t vp[ROWS][EPL], hp[ROWS], cl[ROWS][EPL];
            load_rows(ps, pend_tile, pbase, pstaged, kp, vp, hp);
            const uint32_t *pcl = stage_vals(ps) + seg;
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int j = 0; j < EPL; ++j) cl[r][j] = pcl[(r * EPL + j) * 32 + lane];
            __syncwarp();
            KU *pk = stage_keys(ps) + seg;
            uint32_t *pvals = stage_vals(ps) + seg;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const uint32_t m = pend_info[r] & 0xffu, offc = pend_info[r] >> 8;
                uint32_t q = offc;   // run index - cw of this chunk's first head
                // the open run's value where the chunk starts
                const uint32_t vin = offc ? pend_offv[r] : RunValue<VU>::add(pv, pend_offv[r]);
                bool first = true;
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    if ((m >> j) & 1u) {
                        pk[rbk_sw(q)] = kp[r][j];
                        pvals[rbk_sw(q)] = first ? RunValue<VU>::add(vin, cl[r][j]) : cl[r][j];
                        first = false;
                        ++q;
                    }
                }
            }
            __syncwarp();
            for (uint32_t q = lane; q < pend_rc; q += 32) {
                ukeys[cw + q] = pk[rbk_sw(q)];
                if (cw + q > 0u) aggs[cw + q - 1u] = pvals[rbk_sw(q)];
            }
            // this warp is done with the stage
            __syncwarp();
            if (lane == 0) {
                if (warp == 0) PS_TRACE_POINT(pend_tile, PS_TRACE_STORED);
                mbar_arrive(&empty[ps]);
            }
            pend = false;
        };
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            const int slot = (int)(k % R);
            if (!role_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                abort_meet(&s_abort, 1, CT);
                break;
            }
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) {
                if (pend) write_dense();
                // end marker: pass it on to every look-back and writer warp,
                // on the slots of the next iterations (the producer, which
                // stopped here, writes none of them again)
                if (warp == 0 && lane == 0) {
#pragma unroll
                    for (int i = 0; i < kREnds; ++i) {
                        if (i > 0) tile_of[(k + i) % R] = num_tiles;
                        if (i < kLB) mbar_arrive(&agg_done[(k + i) % R]);
                    }
                }
                __syncwarp();
                if (lane == 0)
#pragma unroll
                    for (int i = 0; i < kRW; ++i) mbar_arrive(&packed[(k + i) % R]);
                break;
            }
            const unsigned long long base = (unsigned long long)tile * TILE;
            const bool staged = a.use_bulk && base + TILE <= n;
            if (warp == 0 && lane == 0) {
                PS_TRACE_POINT(tile, PS_TRACE_DATA);
                PS_TRACE_POINT(tile, PS_TRACE_COMPUTE_START);
            }
            KU kk[ROWS][EPL];
            uint32_t vv[ROWS][EPL];
            uint32_t hm[ROWS];
            load_rows(s, tile, base, staged, kk, vv, hm);
            // Segmented inclusive scan of the chunk pairs over the lanes, the
            // rows side by side so that their shuffle chains overlap.  A
            // chunk's pair is (its heads, its value from its last head on);
            // the segment of lane l starts at the nearest lane <= l whose
            // chunk holds a head (none: it reaches back past lane 0), and a
            // partial from lane l-d joins only while l-d lies in it.
            uint32_t offc[ROWS], offv[ROWS];   // exclusive pair of the chunk within the warp
            uint32_t rc = 0u, rv = 0u;         // pair of the warp's rows so far
            // Each head's closing value -- the value of the run it closes,
            // summed from the chunk's start at most -- goes to the warp's
            // slice of the stage's values, entry (r * EPL + j) * 32 + lane
            // (consecutive lanes, consecutive words): the pack then visits
            // the heads only.  The warp's values are all in registers first.
            uint32_t *cls = stage_vals(s) + seg;
            __syncwarp();
            {
                uint32_t cc[ROWS], cv[ROWS], cnt[ROWS];
                int seg_lo[ROWS];
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    uint32_t v = 0u;
#pragma unroll
                    for (int j = 0; j < EPL; ++j) {
                        const bool h = (hm[r] >> j) & 1u;
                        if (h) cls[(r * EPL + j) * 32 + lane] = v;
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
            }
            P *sw = s_warp[k & 1];
            if (lane == 0) sw[warp] = pair_of(rc, rv);
            named_barrier(1, CT);   // every warp has read the stage and posted its pair
            if (aborted(&s_abort)) break;
            // the warps' pairs scanned across lanes 0 .. kRCW-1 (earlier part
            // on the left): the pair of the tile's elements before this
            // warp's, and the tile's
            P wp = lane < kRCW ? sw[lane] : (P)0;
#pragma unroll
            for (int d = 1; d < kRCW; d <<= 1) {
                const P o = __shfl_up_sync(kFull, wp, d);
                if (lane >= d) wp = Op::combine(o, wp);
            }
            const P agg = __shfl_sync(kFull, wp, kRCW - 1);
            P wex = __shfl_sync(kFull, wp, warp > 0 ? warp - 1 : 0);
            if (warp == 0) wex = 0;
            const bool sparse = pair_count(agg) <= (uint32_t)CAP;
            if (warp == 0 && lane == 0) {
                // A at once (P for tile 0, whose exclusive pair is empty)
                Desc<P, 2>::store(desc, tile, tile == 0 ? kFlagP : kFlagA, agg, epoch);
                PS_TRACE_POINT(tile, PS_TRACE_AGGREGATE);
                agg_of[slot] = agg;
                sparse_of[slot] = sparse ? 1 : 0;
                mbar_arrive(&agg_done[slot]);
            }
            if (sparse) {
                // pack the runs in the iteration's output buffer, once the
                // writer is done with its previous tile; run q of the tile
                // gets its key and the value of the run its head closes,
                // summed from the tile's start at most
                const int o = (int)(k % NOB);
                if (k >= NOB && !role_wait(&ob_empty[o], (uint32_t)((k / NOB - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    abort_meet(&s_abort, 1, CT);
                    break;
                }
                KU *ok = out_keys(o);
                uint32_t *ov = out_vals(o);
                const uint32_t wq0 = pair_count(wex), wv0 = pair_value(wex);
                const KU *ks = stage_keys(s);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    uint32_t q = wq0 + offc[r];
                    // the open run's value where the chunk starts: the chunk's
                    // first head adds it to its closing value
                    uint32_t vin = offc[r] ? offv[r] : RunValue<VU>::add(wv0, offv[r]);
                    const uint32_t e0 = (uint32_t)(seg + (r * 32 + lane) * EPL);
                    for (uint32_t mm = hm[r]; mm; mm &= mm - 1u) {
                        const uint32_t j = (uint32_t)(__ffs(mm) - 1);
                        ok[rbk_sw(q)] = staged ? ks[e0 + j] : keys[base + e0 + j];
                        ov[rbk_sw(q)] = RunValue<VU>::add(vin, cls[((uint32_t)r * EPL + j) * 32 + lane]);
                        vin = 0u;   // later heads' runs begin inside the chunk
                        ++q;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&packed[slot]);
                    mbar_arrive(&empty[s]);   // this warp is done with the stage
                }
            } else {
                // a dense tile: nothing for the writer (it only frees the
                // buffer); the compute warps write it after the next tile's
                // pass, and hand its stage back then
                if (lane == 0) mbar_arrive(&packed[slot]);
            }
            if (pend) write_dense();   // the previous dense tile, now that this tile's pair is out
            if (!sparse) {
                pend = true;
                pend_at = (uint32_t)s | ((uint32_t)slot << 8) | ((uint32_t)((k / R) & 1) << 16);
                pend_tile = (uint32_t)tile;
                pend_wex = wex;
                pend_rc = rc;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    pend_info[r] = hm[r] | (offc[r] << 8);
                    pend_offv[r] = offv[r];
                }
            }
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
    long long grid = (long long)sms * kRCtasPerSm;
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
