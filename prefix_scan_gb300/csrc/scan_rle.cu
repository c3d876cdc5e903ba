// scan_rle.cu -- single-pass run-length encoding (decoupled look-back paper
// summary, A5: run-length encoding among the fused compaction workloads).
//
// Element i opens a run ("head") when i == 0 or its key bits differ from
// those of element i-1.  Run c is the c-th head in input order; its length
// is the distance from its head to the next one (to n for the last run).
// So the encoding is a selection of the heads, positioned by the exclusive
// count of heads before them, where each head also closes the run before
// it:   unique_keys[c] = key_i,   counts[c-1] = i - (position of head c-1).
//
// The scan state of a prefix is the pair (heads in it, position of its last
// head), combined as (sum of counts, larger position): positions grow along
// the input, so the later part's last head wins whenever it has one, and a
// part without heads carries position 0 -- the same as "the last head is
// element 0", which is what a prefix whose only head is element 0 means.
// The operator is commutative, so the look-back folds its window with the
// butterfly reduction.  The pair travels as one 64-bit word,
// count << 32 | position, in the two-word descriptor of the int64 scan.
//
// Reduce-by-key needs the segmented sum of the values and keeps its own
// kernel (scan_reduce_by_key.cu); lengths need none: a length is a
// difference of two head positions.
//
// Structure as in the persistent scan and the select kernel: a producer warp
// takes tile ids and bulk-copies the tile's keys -- starting one 16-byte
// vector early, so the key before the tile (the "halo") is in shared memory
// too -- into a 3-stage ring; two aggregator warps count the heads of half
// the tile each and find the last one, and the second to finish publishes
// the tile's pair; a look-back warp resolves the tile's exclusive pair;
// eight compute warps find the heads of their rows, count them with warp
// scans and write each head's key and the length of the run it closes.  A
// warp with few heads writes them straight from registers and hands the
// stage back as soon as the keys are in registers; a warp dense in heads
// packs each row's runs in its slice of the stage first, so that they go out
// as contiguous ranges.  Counts and positions are 32-bit (n < 2^32).
#include "scan_device.cuh"
#include "scan_pipeline.cuh"
#include "scan_trace.cuh"

namespace ps {

namespace {

constexpr int kLCW = kThreads / 32;   // compute warps per CTA
constexpr int kLStages = 3;
constexpr int kLRing = 2 * kLStages;  // hand-off slots: iteration k uses k % kLRing
// Aggregator warps: each reduces an equal part of a tile.  One warp took
// about 2 us per 32 KiB tile, which capped each CTA at one tile per
// aggregation; twelve warps of 80 registers still fit two CTAs per SM.
#ifndef PS_RLE_AGG_WARPS
#define PS_RLE_AGG_WARPS 2
#endif
constexpr int kLAgg = PS_RLE_AGG_WARPS;
// Look-back warps; warp j resolves iterations j, j + LB, ...  (a macro so
// that a tuning sweep can rebuild).
#ifndef PS_RLE_LOOKBACK_WARPS
#define PS_RLE_LOOKBACK_WARPS 1
#endif
constexpr int kLLB = PS_RLE_LOOKBACK_WARPS;
static_assert(kLRing % kLLB == 0, "the look-back warps step through the ring evenly");
constexpr int kLThreads = (kLCW + 1 + kLLB + kLAgg) * 32;   // compute, producer, look-back, aggregators

// Role waits suspend in the barrier for up to this many nanoseconds per try
// (0: poll), so that waiting warps leave the issue slots to working ones; a
// macro so that a tuning sweep can rebuild.
#ifndef PS_RLE_WAIT_NS
#define PS_RLE_WAIT_NS 2000
#endif
// A warp whose 32 x ITEMS keys hold more heads than this packs each row's
// runs in its slice of the stage and writes them out as contiguous ranges;
// below it, each head is written straight from registers.
#ifndef PS_RLE_DENSE_HEADS
#define PS_RLE_DENSE_HEADS 128
#endif
// Position of packed entry q in a warp's slice: XOR-swizzled within each 32
// entries, so that lanes packing entries 8 apart (every key a head) and
// lanes reading 32 consecutive entries hit distinct banks.
__device__ __forceinline__ uint32_t rle_sw(uint32_t q) { return q ^ ((q >> 5) & 7u); }
__device__ __forceinline__ bool rle_wait(uint64_t *bar, uint32_t parity) {
    return PS_RLE_WAIT_NS ? mbar_wait_suspend(bar, parity, PS_RLE_WAIT_NS) : mbar_wait(bar, parity);
}

// k[j] for a j known only at run time, without local memory: a tree of
// selects on the bits of j (E - 1 selects on log2(E) bit tests).
template <typename KU, int E>
__device__ __forceinline__ KU pick(const KU (&k)[E], int j) {
    static_assert(E == 4 || E == 8, "four or eight keys");
    const bool b0 = j & 1, b1 = j & 2;
    const KU a0 = b0 ? k[1] : k[0], a1 = b0 ? k[3] : k[2];
    const KU lo = b1 ? a1 : a0;
    if constexpr (E == 4) {
        return lo;
    } else {
        const KU a2 = b0 ? k[5] : k[4], a3 = b0 ? k[7] : k[6];
        const KU hi = b1 ? a3 : a2;
        return (j & 4) ? hi : lo;
    }
}

// (heads << 32 | position of the last head); `a` is the earlier part.
struct OpRle {
    static constexpr bool kCommutative = true;
    template <typename U> static __device__ __forceinline__ U identity() { return U(0); }
    template <typename U> static __device__ __forceinline__ U combine(U a, U b) {
        const uint32_t pa = (uint32_t)a, pb = (uint32_t)b;
        return (((a >> 32) + (b >> 32)) << 32) | (pa > pb ? pa : pb);
    }
};

// 16-byte key vectors: four 32-bit keys or two 64-bit keys.
template <typename KU> struct RleVec;
template <> struct RleVec<uint32_t> {
    using V = uint4;
    static constexpr int N = 4;
    static __device__ __forceinline__ uint32_t key(const V &v, int j) { return vget(v, j); }
};
template <> struct RleVec<unsigned long long> {
    using V = ulonglong2;
    static constexpr int N = 2;
    static __device__ __forceinline__ unsigned long long key(const V &v, int j) { return vget(v, j); }
};

// 32 KiB of keys per tile, plus the halo vector in front of them.
// Bytes of keys per tile (a macro so that a tuning sweep can rebuild).
#ifndef PS_RLE_TILE_BYTES
#define PS_RLE_TILE_BYTES 32768
#endif
template <typename KU> constexpr long long rle_tile() { return PS_RLE_TILE_BYTES / (long long)sizeof(KU); }
template <typename KU> constexpr uint32_t rle_stage_bytes() { return (uint32_t)(rle_tile<KU>() * sizeof(KU) + 16); }
template <typename KU> constexpr size_t rle_smem_bytes() {
    return (size_t)kLStages * rle_stage_bytes<KU>() +
           ((size_t)kLStages * 2 * 8 + (size_t)kLRing * (2 * 8 + 8 + 8 + 8) + 127) / 128 * 128;
}

}  // namespace


template <typename KU>
__global__ void __launch_bounds__(kLThreads, kPCtasPerSm)
rle_kernel(RbkArgs a, long long num_tiles) {
    using KV = RleVec<KU>;
    using V = typename KV::V;
    using P = unsigned long long;
    constexpr int VK = KV::N;
    constexpr long long TILE = rle_tile<KU>();
    constexpr int ITEMS = (int)(TILE / kThreads);   // keys per compute lane
    constexpr int EPL = 2 * VK;                     // keys per lane per row: two vectors
    constexpr int ROWS = ITEMS / EPL;
    constexpr int S = kLStages, R = kLRing;
    constexpr uint32_t KEY_BYTES = (uint32_t)(TILE * sizeof(KU));
    constexpr uint32_t STAGE = rle_stage_bytes<KU>();
    constexpr int NV = (int)(TILE / VK);   // vectors per tile
    constexpr int CT = kLCW * 32;
    static_assert(ITEMS % EPL == 0 && NV % 32 == 0 && STAGE % 16 == 0, "tile geometry");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * STAGE);
    uint64_t *empty = full + S;
    uint64_t *agg_done = empty + S;   // the rest: R slots, slot k % R
    uint64_t *prefix_ready = agg_done + R;
    long long *tile_of = reinterpret_cast<long long *>(prefix_ready + R);
    P *agg_of = reinterpret_cast<P *>(tile_of + R);
    P *excl_of = agg_of + R;
    __shared__ P s_warp[2][kLCW];
    __shared__ int s_abort;   // a compute warp's wait ran out: all of them leave
    __shared__ P s_part[kLRing][kLAgg];   // the aggregators' parts of a tile's pair
    __shared__ int s_parts_done[kLRing];  // parts in: the last one publishes
    // stage s: [halo vector][TILE keys]
    auto stage_keys = [&](int s) { return reinterpret_cast<KU *>(smem + (size_t)s * STAGE + 16); };

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Header *hdr = reinterpret_cast<Header *>(a.ws);
    void *desc = a.ws + kHeaderBytes;
    const unsigned long long n = a.n;
    const KU *keys = reinterpret_cast<const KU *>(a.keys);
    KU *ukeys = reinterpret_cast<KU *>(a.unique_keys);
    uint32_t *counts = reinterpret_cast<uint32_t *>(a.aggs);

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
            mbar_init(&empty[s], kLCW + kLAgg);   // compute warps + aggregators
        }
        for (int slot = 0; slot < R; ++slot) {
            mbar_init(&agg_done[slot], 1);
            mbar_init(&prefix_ready[slot], 1);
            tile_of[slot] = num_tiles;   // end marker until the producer fills it
            s_parts_done[slot] = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!s_ok) return;   // same verdict in every CTA
    const uint32_t epoch = s_epoch;
    if (tid == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_HEADER);

    if (warp == kLCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int ends = 0;   // end markers sent: one per look-back warp
            for (long long k = 0;; ++k) {
                const int s = (int)(k % S);
                if (k >= S && !rle_wait(&empty[s], (uint32_t)((k / S - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    break;
                }
                const long long t = ends ? num_tiles : (long long)atomicAdd(&hdr->tile_counter, 1ull);
                tile_of[k % R] = t;
                if (t < num_tiles) {
                    prefetch_descriptor<2>(desc, t);
                    PS_TRACE_POINT(t, PS_TRACE_CLAIM);
                    PS_TRACE_CTA(t);
                }
                if (a.use_bulk && t < num_tiles && (unsigned long long)(t + 1) * TILE <= n) {
                    if (t == 0) {
                        mbar_arrive_expect_tx(&full[s], KEY_BYTES);
                        bulk_load(stage_keys(s), keys, KEY_BYTES, &full[s]);
                    } else {
                        mbar_arrive_expect_tx(&full[s], KEY_BYTES + 16u);
                        bulk_load(stage_keys(s) - VK, keys + t * TILE - VK, KEY_BYTES + 16u, &full[s]);
                    }
                } else {
                    mbar_arrive(&full[s]);   // end marker, or a tile read from global
                }
                if (t >= num_tiles && ++ends == kLLB) break;
            }
            if (epoch != kEpochMask) claims_done(hdr, a.ws_bytes, epoch);
        }
    } else if (warp > kLCW && warp <= kLCW + kLLB) {
        // ---------------- look-back warps: the tile's exclusive pair ----------------
        for (long long k = warp - (kLCW + 1);; k += kLLB) {
            const int slot = (int)(k % R);
            if (!rle_wait(&agg_done[slot], (uint32_t)((k / R) & 1))) {
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
                excl = look_back<P, 2, kLookbackK, OpRle>(desc, tile, epoch, a.max_polls, &hdr->status,
                                                          PS_TRACE_LOOKBACK(tile));
                if (lane == 0) Desc<P, 2>::store(desc, tile, kFlagP, OpRle::combine(excl, agg), epoch);
            }
            if (lane == 0) {
                if (tile == num_tiles - 1) {
                    // the whole input: the number of runs and the last head,
                    // whose run ends at n
                    const P incl = OpRle::combine(excl, agg);
                    const uint32_t runs = (uint32_t)(incl >> 32);
                    if (runs > 0) counts[runs - 1] = (uint32_t)(n - (uint32_t)incl);
                    if (a.num_runs) *a.num_runs = runs;
                }
                excl_of[slot] = excl;
                PS_TRACE_POINT(tile, PS_TRACE_PREFIX);
                mbar_arrive(&prefix_ready[slot]);
            }
        }
    } else if (warp > kLCW + kLLB) {
        // ---------------- aggregators: the tile's pair, published at once ----------------
        // kLAgg warps, each over an equal part of the tile; the last to
        // finish combines the parts and publishes the pair.
        const int g = warp - (kLCW + 1 + kLLB);
        int ends = 0;   // end markers passed on: one per look-back warp
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!rle_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const int slot = (int)(k % R);
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) {   // end marker: pass it on to a look-back warp
                if (g == 0 && lane == 0) mbar_arrive(&agg_done[slot]);
                if (++ends == kLLB) break;
                continue;
            }
            if (g == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_DATA);
            const unsigned long long base = (unsigned long long)tile * TILE;
            uint32_t heads = 0;
            uint32_t last = 0;   // position of the part's last head (0: none)
            if (a.use_bulk && base + TILE <= n) {
                // lane l takes the C consecutive vectors of its chunk, so
                // the key before a vector is the last key of the one it read
                // before (a register); it visits them from vector r = l mod 8
                // on and wraps round, so that the 8 lanes one 16-byte load
                // serves hit distinct bank groups.  Only two keys come from
                // elsewhere: the one before the chunk (the halo for the
                // tile's first chunk; tile 0 starts with a value that differs
                // from element 0) and the one before vector r, which comes
                // round last.
                constexpr int PV = NV / kLAgg;   // vectors per part
                constexpr int C = PV / 32;
                static_assert(PV % 32 == 0 && C >= 8 && (C & (C - 1)) == 0, "chunk of a power-of-two size >= 8");
                const KU *ks = stage_keys(s);
                const int v_chunk = g * PV + lane * C;   // the chunk's first vector
                const V *kv = reinterpret_cast<const V *>(ks) + v_chunk;
                const int r0 = lane & 7;
                const int e_chunk = v_chunk * VK;   // tile index of the chunk's first key
                const KU before_chunk = (tile == 0 && e_chunk == 0) ? (KU)~ks[0] : ks[e_chunk - 1];
                KU carry = r0 == 0 ? before_chunk : ks[e_chunk + r0 * VK - 1];
                int last_vec = -1;   // highest vector of the chunk that holds a head
#pragma unroll 8
                for (int q = 0; q < C; ++q) {
                    const int vi = (q + r0) & (C - 1);
                    const V x = kv[vi];
                    const KU prev = vi == 0 ? before_chunk : carry;
                    carry = KV::key(x, VK - 1);
                    uint32_t h = 0;
#pragma unroll
                    for (int j = 0; j < VK; ++j) h += (uint32_t)(KV::key(x, j) != (j ? KV::key(x, j - 1) : prev));
                    heads += h;
                    last_vec = (h && vi > last_vec) ? vi : last_vec;
                }
                // the part's last head: in the highest lane that has one, in
                // that lane's highest vector with one (same in every lane)
                const int lv_lane = __reduce_max_sync(kFull, last_vec >= 0 ? lane : -1);
                if (lv_lane >= 0) {
                    const int lv = g * PV + lv_lane * C + __shfl_sync(kFull, last_vec, lv_lane);
                    const V x = reinterpret_cast<const V *>(ks)[lv];
                    const KU prev = lv > 0 ? ks[lv * VK - 1] : tile == 0 ? (KU)~KV::key(x, 0) : ks[-1];
                    uint32_t m = 0;
#pragma unroll
                    for (int j = 0; j < VK; ++j) m |= (uint32_t)(KV::key(x, j) != (j ? KV::key(x, j - 1) : prev)) << j;
                    last = (uint32_t)(base + (unsigned long long)(lv * VK + 31 - __clz(m)));
                }
            } else {
                constexpr long long PART = TILE / kLAgg;
                const unsigned long long lo = base + (unsigned long long)(g * PART);
                const unsigned long long hi = base + (unsigned long long)((g + 1) * PART);
                const unsigned long long end = hi < n ? hi : n;
                long long le = -1;
                for (unsigned long long i = lo + lane; i < end; i += 32)
                    if (i == 0 || keys[i] != keys[i - 1]) { ++heads; le = (long long)(i - base); }
                const int lmax = __reduce_max_sync(kFull, (int)le);
                last = lmax >= 0 ? (uint32_t)(base + (unsigned long long)lmax) : 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            heads = __reduce_add_sync(kFull, heads);
            if (lane == 0) {
                // parts later in the tile have larger positions, so the
                // parts combine in any order
                volatile P *part = s_part[slot];
                part[g] = ((P)heads << 32) | last;
                __threadfence_block();
                if (atomicAdd(&s_parts_done[slot], 1) == kLAgg - 1) {
                    __threadfence_block();
                    P agg = 0;
#pragma unroll
                    for (int gg = 0; gg < kLAgg; ++gg) agg = OpRle::combine(agg, (P)part[gg]);
                    s_parts_done[slot] = 0;   // the slot's next use is kLRing iterations on
                    Desc<P, 2>::store(desc, tile, tile == 0 ? kFlagP : kFlagA, agg, epoch);
                    PS_TRACE_POINT(tile, PS_TRACE_AGGREGATE);
                    agg_of[slot] = agg;
                    mbar_arrive(&agg_done[slot]);
                }
            }
        }
    } else {
        // ---------------- compute warps: find the heads, write the runs ----------------
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!rle_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                abort_meet(&s_abort, 1, CT);
                break;
            }
            const int slot = (int)(k % R);
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            const unsigned long long base = (unsigned long long)tile * TILE;
            const bool staged = a.use_bulk && base + TILE <= n;
            const int seg = warp * 32 * ITEMS;   // the warp's first key in the tile
            if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_COMPUTE_START);

            // Rows of two 16-byte vectors per lane (EPL keys); lanes 4-7 of
            // each quarter-warp read their pair in swapped order, so that
            // the eight 16-byte reads of a quarter-warp fall in distinct bank
            // groups.  Bit j of m[r]: key j of the lane's chunk of row r
            // opens a run.
            KU kk[ROWS][EPL];
            uint32_t m[ROWS];
            if (staged) {
                const KU *ks = stage_keys(s);
                const V *kv = reinterpret_cast<const V *>(ks);
                const int rot = (lane >> 2) & 1;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const int e0 = seg + (r * 32 + lane) * EPL;
                    const V x0 = kv[e0 / VK + rot], x1 = kv[e0 / VK + (rot ^ 1)];
                    const V lo = rot ? x1 : x0, hi = rot ? x0 : x1;
#pragma unroll
                    for (int j = 0; j < VK; ++j) {
                        kk[r][j] = KV::key(lo, j);
                        kk[r][VK + j] = KV::key(hi, j);
                    }
                    KU prev = __shfl_up_sync(kFull, kk[r][EPL - 1], 1);
                    if (lane == 0) prev = ks[e0 - 1];   // e0 == 0 reads the halo
                    uint32_t mm = 0;
#pragma unroll
                    for (int j = 0; j < EPL; ++j) mm |= (uint32_t)(kk[r][j] != (j ? kk[r][j - 1] : prev)) << j;
                    if (tile == 0 && e0 == 0) mm |= 1u;
                    m[r] = mm;
                }
            } else {
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    uint32_t mm = 0;
#pragma unroll
                    for (int j = 0; j < EPL; ++j) {
                        const unsigned long long i = base + seg + (unsigned long long)((r * 32 + lane) * EPL + j);
                        kk[r][j] = i < n ? keys[i] : KU(0);
                        mm |= (uint32_t)(i < n && (i == 0 || kk[r][j] != keys[i - 1])) << j;
                    }
                    m[r] = mm;
                }
            }
            // The keys are in registers.  A sparse warp does not touch the
            // stage again and hands it back before the tile's pair arrives
            // (the hand-off ring keeps the slots apart); a dense one packs
            // its runs in its slice of the stage -- free once the pair has
            // arrived, since the aggregator finished reading the stage before
            // the look-back began -- and hands it back after writing them.
            uint32_t wh = 0;
#pragma unroll
            for (int r = 0; r < ROWS; ++r) wh += (uint32_t)__popc(m[r]);
            const bool dense = __reduce_add_sync(kFull, wh) > (uint32_t)PS_RLE_DENSE_HEADS;
            __syncwarp();
            if (!dense && lane == 0) mbar_arrive(&empty[s]);

            // Per row: heads before each lane's chunk (warp scan of the
            // chunk counts), and the position of the last head before it --
            // in the nearest lower lane that has one (ballot + one shuffle),
            // else in an earlier row of this warp.  Both are below the warp's
            // 32 * ITEMS keys, so a row's mask, count and previous head share
            // one word (registers are at the cap that two CTAs per SM allow):
            //   bits 0-7 mask, 8-18 heads before, 19-29 previous head (offset
            //   from the warp's first key), bit 30 set if that head exists.
            static_assert(32 * ITEMS <= 2048 && EPL <= 8, "row words hold 8 mask bits and two 11-bit fields");
            const uint32_t lt_mask = (1u << lane) - 1u;
            const uint32_t wbase = (uint32_t)(base + (unsigned long long)seg);   // position of the warp's first key
            uint32_t info[ROWS];
            uint32_t run_c = 0, run_p = 0, run_has = 0;   // heads so far in this warp, the last one
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const uint32_t t = (uint32_t)__popc(m[r]);
                const uint32_t sc = warp_inclusive<uint32_t>(t, lane);
                const uint32_t before = run_c + (sc - t);
                run_c += __shfl_sync(kFull, sc, 31);
                const uint32_t lp = m[r] ? (uint32_t)((r * 32 + lane) * EPL + 31 - __clz(m[r])) : 0u;
                const uint32_t hb = __ballot_sync(kFull, m[r] != 0u);
                const uint32_t below = hb & lt_mask;
                const uint32_t from = __shfl_sync(kFull, lp, below ? 31 - __clz(below) : 0);
                const uint32_t pp = below ? from : run_p;
                const uint32_t has = below ? 1u : run_has;
                info[r] = m[r] | (before << 8) | (pp << 19) | (has << 30);
                const uint32_t row_last = __shfl_sync(kFull, lp, hb ? 31 - __clz(hb) : 0);
                run_p = hb ? row_last : run_p;
                run_has = hb ? 1u : run_has;
            }
            run_p = run_has ? wbase + run_p : 0u;   // as a position, 0 for none
            P *sw = s_warp[k & 1];
            if (lane == 0) sw[warp] = ((P)run_c << 32) | run_p;
            named_barrier(1, CT);
            if (aborted(&s_abort)) break;
            P warp_excl = 0;
#pragma unroll
            for (int w = 0; w < kLCW; ++w)
                if (w < warp) warp_excl = OpRle::combine(warp_excl, sw[w]);
            if (!rle_wait(&prefix_ready[slot], (uint32_t)((k / R) & 1)))
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
            const P pre = OpRle::combine(excl_of[slot], warp_excl);
            const uint32_t cw = (uint32_t)(pre >> 32), pw = (uint32_t)pre;
            if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_PREFIX_RECEIVED);

            if (!dense) {
                // each head: its key to unique_keys[c], and the length of run
                // c - 1 (which it closes) to counts[c - 1]; only the set bits
                // of the mask are visited
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint32_t w = info[r];
                    const uint32_t pos0 = wbase + (uint32_t)((r * 32 + lane) * EPL);
                    uint32_t c = cw + ((w >> 8) & 0x7ffu);
                    uint32_t prev = (w >> 30) ? wbase + ((w >> 19) & 0x7ffu) : pw;
                    for (uint32_t mm = w & 0xffu; mm; mm &= mm - 1u) {
                        const int j = __ffs(mm) - 1;
                        const KU key = pick<KU, EPL>(kk[r], j);
                        ukeys[c] = key;
                        if (c > 0u) counts[c - 1u] = pos0 + (uint32_t)j - prev;
                        prev = pos0 + (uint32_t)j;
                        ++c;
                    }
                }
            } else {
                // per row: the row's runs are the contiguous run indices
                // [cw + first, cw + first + nh); pack each head's key and
                // offset in order, then write keys and lengths (differences
                // of consecutive head offsets) with consecutive lanes on
                // consecutive entries
                KU *pk = stage_keys(s) + seg;                                      // 32 * EPL keys
                uint32_t *pp = reinterpret_cast<uint32_t *>(pk + 32 * EPL);        // 32 * EPL offsets
                static_assert(32 * EPL * (sizeof(KU) + 4) <= 32 * ITEMS * sizeof(KU), "a row's runs fit the slice");
                uint32_t row_prev = pw;   // position of the last head before the row
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const uint32_t w = info[r];
                    const uint32_t rb = (w >> 8) & 0x7ffu;
                    const uint32_t first = __shfl_sync(kFull, rb, 0);
                    const uint32_t nh = __shfl_sync(kFull, rb + (uint32_t)__popc(w & 0xffu), 31) - first;
                    uint32_t q = rb - first;
                    for (uint32_t mm = w & 0xffu; mm; mm &= mm - 1u) {
                        const int j = __ffs(mm) - 1;
                        const KU key = pick<KU, EPL>(kk[r], j);
                        pk[rle_sw(q)] = key;
                        pp[rle_sw(q)] = (uint32_t)((r * 32 + lane) * EPL + j);
                        ++q;
                    }
                    __syncwarp();
                    const uint32_t c0 = cw + first;
                    for (uint32_t t = lane; t < nh; t += 32) {
                        const uint32_t pos = wbase + pp[rle_sw(t)];
                        const uint32_t pv = t ? wbase + pp[rle_sw(t - 1u)] : row_prev;
                        ukeys[c0 + t] = pk[rle_sw(t)];
                        if (c0 + t > 0u) counts[c0 + t - 1u] = pos - pv;
                    }
                    if (nh) row_prev = wbase + pp[rle_sw(nh - 1u)];
                    __syncwarp();
                }
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_STORED);
        }
        if (warp == 0 && lane == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_DONE);
    }

    // the last producer readied the workspace; before an epoch wrap the
    // last CTA to finish does
    if (epoch == kEpochMask) finish_call(hdr, a.ws, a.ws_bytes, epoch);
}

template <typename KU>
static cudaError_t launch_rle_keys(const RbkArgs &a, cudaStream_t s) {
    constexpr size_t smem = rle_smem_bytes<KU>();
    const long long tiles = (long long)((a.n + rle_tile<KU>() - 1) / rle_tile<KU>());
    static volatile int configured[64] = {};
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(rle_kernel<KU>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    long long grid = (long long)sms * kPCtasPerSm;
    if (grid > tiles) grid = tiles;
    rle_kernel<KU><<<(unsigned int)grid, kLThreads, smem, s>>>(a, tiles);
    return cudaGetLastError();
}

cudaError_t launch_run_length_encode(const RbkArgs &a, ps_dtype key_dt, cudaStream_t s) {
    // the workspace is sized for reduce-by-key's tiles, which are no larger
    static_assert(rle_tile<uint32_t>() >= (long long)rbk_tile_elems(PS_INT32) &&
                  rle_tile<unsigned long long>() >= (long long)rbk_tile_elems(PS_INT64),
                  "run-length encoding must need no more descriptors than reduce-by-key");
    return key_dt == PS_INT64 ? launch_rle_keys<unsigned long long>(a, s) : launch_rle_keys<uint32_t>(a, s);
}

TRACE_COPY_FUNCTIONS(trace_copy_rle, trace_copy_rle_ctas)

}  // namespace ps
