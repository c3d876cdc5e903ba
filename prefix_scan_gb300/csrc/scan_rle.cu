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
// Roles.  A producer warp takes tile ids and bulk-copies each tile's keys --
// starting one 16-byte vector early, so the key before the tile (the "halo")
// is in shared memory too -- into a ring of stages.  The compute warps
// (sixteen: one CTA per SM and 64 KiB tiles, so that every look-back covers
// twice the bytes it did with two CTAs of 32 KiB tiles) take the tiles in
// order and never wait for a tile's
// prefix: each lane finds the heads among 128 consecutive bytes of keys (one
// mask), a warp scan and a scan of the warps' totals count them, the warps
// publish the tile's pair (A; P for tile 0) themselves and pack the tile's
// runs into an output buffer -- each head's key, read back from the stage,
// and its 16-bit position within the tile, in order -- after which the stage
// goes straight back to the producer.  Look-back warps resolve each tile's
// exclusive pair; writer warps wait for it and write the buffer out as
// contiguous ranges (keys, and lengths as differences of consecutive head
// positions), then free the buffer.  So a stage is held only from its copy
// to the compute warps' pass, and the look-back's latency stays off both the
// stages and the compute warps: it is covered by the output buffers, which
// hold a few bytes per head.  A tile with more heads than a buffer holds (a
// dense tile) is written by the compute warps themselves -- all of them
// instead of one for a tile that writes as much as it reads -- one iteration
// late: they publish its pair, keep its stage, do the next tile's pass (so
// that tile's pair is published too), and only then wait for the dense
// tile's prefix, re-read its keys from the stage, pack each row's runs in
// their slice of the stage (the head masks kept from the pass) and write
// them as contiguous ranges.  Waiting for a tile's prefix before publishing
// the next tile's pair would chain every CTA's tiles behind the look-backs
// of its earlier ones.  Counts and positions are 32-bit (n < 2^32).
#include "scan_device.cuh"
#include "scan_pipeline.cuh"
#include "scan_trace.cuh"

namespace ps {

namespace {

// Compute warps per CTA and CTAs per SM (macros, so that a tuning sweep can
// rebuild); a tile is 128 bytes of keys per compute lane.
#ifndef PS_RLE_COMPUTE_WARPS
#define PS_RLE_COMPUTE_WARPS 16
#endif
#ifndef PS_RLE_CTAS_PER_SM
#define PS_RLE_CTAS_PER_SM 1
#endif
constexpr int kLCW = PS_RLE_COMPUTE_WARPS;
constexpr int kLCtasPerSm = PS_RLE_CTAS_PER_SM;
static_assert(kLCW >= 1 && kLCW <= 32, "the warps' pairs are scanned across the lanes of one warp");
// Stages of keys (one tile each) and output buffers (a macro each, so that a
// tuning sweep can rebuild).
#ifndef PS_RLE_STAGES
#define PS_RLE_STAGES 3
#endif
#ifndef PS_RLE_OUT_BUFFERS
#define PS_RLE_OUT_BUFFERS 4
#endif
#ifndef PS_RLE_OUT_BYTES
#define PS_RLE_OUT_BYTES 8192
#endif
// Descriptors per lane in the look-back window (the operator is commutative).
#ifndef PS_RLE_LOOKBACK_K
#define PS_RLE_LOOKBACK_K PS_LOOKBACK_K
#endif
// Look-back warps (warp j resolves iterations j, j + LB, ...) and writer
// warps (the same, for the write-out).
#ifndef PS_RLE_LOOKBACK_WARPS
#define PS_RLE_LOOKBACK_WARPS 2
#endif
#ifndef PS_RLE_WRITER_WARPS
#define PS_RLE_WRITER_WARPS 2
#endif
constexpr int kLStages = PS_RLE_STAGES;
constexpr int kLOut = PS_RLE_OUT_BUFFERS;
constexpr int kLOutBytes = PS_RLE_OUT_BYTES;
constexpr int kLLB = PS_RLE_LOOKBACK_WARPS;
constexpr int kLW = PS_RLE_WRITER_WARPS;
constexpr int cmax(int a, int b) { return a > b ? a : b; }
// Iterations past the end that the compute warps mark: every look-back and
// writer warp waits on its next iteration.
constexpr int kLEnds = cmax(kLLB, kLW);
// Hand-off slots (tile id, pair, exclusive pair, buffer kind and the
// agg_done / prefix_ready / packed mbarriers): iteration k uses slot k % R.
// A slot is reused only after every role is done with it: the writer is at
// most kLOut iterations behind the compute warps (each waits for its buffer
// before a sparse tile), the producer at most kLStages + 1 ahead of their
// pass, and the compute warps write the end markers of up to kLEnds
// iterations ahead.
constexpr int ring_slots() {
    const int need = cmax(kLStages + kLOut + 1, kLEnds + kLOut);
    return (need + 1) / 2 * 2;
}
constexpr int kLRing = ring_slots();
constexpr int kLThreads = (kLCW + 1 + kLLB + kLW) * 32;   // compute, producer, look-back, writer
static_assert(kLStages >= 2, "a dense tile keeps its stage while the next one is scanned");

// Role waits suspend in the barrier for up to this many nanoseconds per try
// (0: poll), so that waiting warps leave the issue slots to working ones; a
// macro so that a tuning sweep can rebuild.
#ifndef PS_RLE_WAIT_NS
#define PS_RLE_WAIT_NS 2000
#endif
// Position of packed entry q in an output buffer or a dense tile's slice:
// XOR-swizzled within each 32 entries, so that lanes packing a row's runs 8
// apart (a dense tile's row where every key is a head) and lanes reading 32
// consecutive entries hit distinct banks.
__device__ __forceinline__ uint32_t rle_sw(uint32_t q) { return q ^ ((q >> 5) & 7u); }
__device__ __forceinline__ bool rle_wait(uint64_t *bar, uint32_t parity) {
    return PS_RLE_WAIT_NS ? mbar_wait_suspend(bar, parity, PS_RLE_WAIT_NS) : mbar_wait(bar, parity);
}

// Key J of the vector in register slot `slot` (known only at run time), by a
// tree of selects on the slot's bits.
template <typename KU, int VK, int J>
__device__ __forceinline__ KU pick_slot(const KU (&k)[8][VK], int slot) {
    const bool b0 = slot & 1, b1 = slot & 2;
    const KU a0 = b0 ? k[1][J] : k[0][J], a1 = b0 ? k[3][J] : k[2][J];
    const KU a2 = b0 ? k[5][J] : k[4][J], a3 = b0 ? k[7][J] : k[6][J];
    const KU lo = b1 ? a1 : a0, hi = b1 ? a3 : a2;
    return (slot & 4) ? hi : lo;
}

// A lane's head mask from slot order to key order: the KPL-bit mask rotated
// left by `sh` bits (slot v holds the lane's vector (v + rot) & 7).
template <int KPL> __device__ __forceinline__ uint32_t rle_unrotate(uint32_t m, int sh) {
    static_assert(KPL == 32 || KPL == 16, "32 or 16 keys per lane");
    if constexpr (KPL == 32) {
        return __funnelshift_l(m, m, sh);
    } else {
        const uint32_t x = m | (m << 16);   // period 16: a 32-bit rotation rotates each half
        return __funnelshift_l(x, x, sh) & 0xffffu;
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

// Bytes of keys per tile: 128 per compute lane.
constexpr long long kLTileBytes = (long long)kLCW * 32 * 128;
template <typename KU> constexpr long long rle_tile() { return kLTileBytes / (long long)sizeof(KU); }
template <typename KU> constexpr uint32_t rle_stage_bytes() { return (uint32_t)(rle_tile<KU>() * sizeof(KU) + 16); }
// Runs an output buffer holds: a key and a 16-bit position within the tile
// each, a multiple of 32 entries (the swizzle stays within each 32).
template <typename KU> constexpr int rle_out_cap() {
    return (int)((kLOutBytes / (sizeof(KU) + 2)) / 32 * 32);
}
template <typename KU> constexpr size_t rle_smem_bytes() {
    return (size_t)kLStages * rle_stage_bytes<KU>() + (size_t)kLOut * kLOutBytes +
           ((size_t)kLStages * 2 * 8 + (size_t)kLOut * 8 + (size_t)kLRing * (3 * 8 + 8 + 8 + 8 + 8) + 127) / 128 *
               128;
}

}  // namespace


template <typename KU>
__global__ void __launch_bounds__(kLThreads, kLCtasPerSm)
rle_kernel(RbkArgs a, long long num_tiles) {
    using KV = RleVec<KU>;
    using V = typename KV::V;
    using P = unsigned long long;
    constexpr int VK = KV::N;
    constexpr long long TILE = rle_tile<KU>();
    constexpr int ITEMS = (int)(TILE / (kLCW * 32));   // keys per compute lane
    constexpr int KPL = 8 * VK;                     // a lane's keys in the pass: eight vectors
    static_assert(ITEMS == KPL, "a lane's keys are 128 bytes");
    constexpr int EPL = 2 * VK;                     // keys per lane per row of a dense write: two vectors
    constexpr int ROWS = ITEMS / EPL;
    constexpr int S = kLStages, R = kLRing, NOB = kLOut;
    constexpr uint32_t KEY_BYTES = (uint32_t)(TILE * sizeof(KU));
    constexpr uint32_t STAGE = rle_stage_bytes<KU>();
    constexpr int CT = kLCW * 32;
    constexpr int CAP = rle_out_cap<KU>();
    static_assert(ITEMS % EPL == 0 && STAGE % 16 == 0 && TILE <= 65536, "tile geometry (16-bit positions)");
    static_assert(CAP >= 32, "output buffer geometry");
    // a dense tile's runs of one row, packed in the warp's slice of the stage
    static_assert(32 * EPL * (sizeof(KU) + 4) <= 32 * ITEMS * sizeof(KU), "a row's runs fit the slice");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *outbuf = smem + (size_t)S * STAGE;
    uint64_t *full = reinterpret_cast<uint64_t *>(outbuf + (size_t)NOB * kLOutBytes);
    uint64_t *empty = full + S;
    uint64_t *ob_empty = empty + S;
    uint64_t *agg_done = ob_empty + NOB;   // the rest: R slots, slot k % R
    uint64_t *prefix_ready = agg_done + R;
    uint64_t *packed = prefix_ready + R;
    long long *tile_of = reinterpret_cast<long long *>(packed + R);
    P *agg_of = reinterpret_cast<P *>(tile_of + R);
    P *excl_of = agg_of + R;
    int *sparse_of = reinterpret_cast<int *>(excl_of + R);
    __shared__ P s_warp[2][kLCW];
    __shared__ int s_abort;   // a compute warp's wait ran out: all of them leave
    // stage s: [halo vector][TILE keys]
    auto stage_keys = [&](int s) { return reinterpret_cast<KU *>(smem + (size_t)s * STAGE + 16); };
    // output buffer o: a sparse tile's runs, CAP keys then CAP positions
    // (within the tile), entry q at rle_sw(q)
    auto out_keys = [&](int o) { return reinterpret_cast<KU *>(outbuf + (size_t)o * kLOutBytes); };
    auto out_pos = [&](int o) {
        return reinterpret_cast<uint16_t *>(outbuf + (size_t)o * kLOutBytes + (size_t)CAP * sizeof(KU));
    };

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
            mbar_init(&empty[s], kLCW);  // each compute warp once it is done with the stage
        }
        for (int o = 0; o < NOB; ++o) mbar_init(&ob_empty[o], 1);   // the writer
        for (int slot = 0; slot < R; ++slot) {
            mbar_init(&agg_done[slot], 1);
            mbar_init(&prefix_ready[slot], 1);
            mbar_init(&packed[slot], kLCW);
            tile_of[slot] = num_tiles;   // end marker until the producer fills it
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
            for (long long k = 0;; ++k) {
                const int s = (int)(k % S);
                if (k >= S && !rle_wait(&empty[s], (uint32_t)((k / S - 1) & 1))) {
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
                if (t >= num_tiles) break;   // the compute warps pass the end marker on
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
                excl = look_back<P, 2, PS_RLE_LOOKBACK_K, OpRle>(desc, tile, epoch, a.max_polls, &hdr->status,
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
        // ---------------- writer warps: a tile's runs, once its pair is known ----------------
        for (long long k = warp - (kLCW + 1 + kLLB);; k += kLW) {
            const int slot = (int)(k % R);
            const uint32_t par = (uint32_t)((k / R) & 1);
            if (!rle_wait(&packed[slot], par)) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            if (!rle_wait(&prefix_ready[slot], par)) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const int o = (int)(k % NOB);
            const unsigned long long base = (unsigned long long)tile * TILE;
            const bool sparse = sparse_of[slot] != 0;
            if (sparse && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_PREFIX_RECEIVED);
            const P excl = excl_of[slot];
            const uint32_t c0 = (uint32_t)(excl >> 32), p0 = (uint32_t)excl;
            const uint32_t tbase = (uint32_t)base;
            if (sparse) {
                // the runs in order: keys to unique_keys[c0 + t], and the
                // length of the run each head closes to counts[c0 + t - 1]
                const uint32_t h = (uint32_t)(agg_of[slot] >> 32);
                const KU *ok = out_keys(o);
                const uint16_t *op = out_pos(o);
                for (uint32_t t = lane; t < h; t += 32) {
                    const uint32_t pos = tbase + op[rle_sw(t)];
                    const uint32_t pv = t ? tbase + op[rle_sw(t - 1u)] : p0;
                    ukeys[c0 + t] = ok[rle_sw(t)];
                    if (c0 + t > 0u) counts[c0 + t - 1u] = pos - pv;
                }
            }   // a dense tile: the compute warps write it
            __syncwarp();
            if (lane == 0) {
                if (sparse) PS_TRACE_POINT(tile, PS_TRACE_STORED);
                mbar_arrive(&ob_empty[o]);
            }
        }
    } else {
        // ---------------- compute warps: find the heads, pack the runs ----------------
        // Lane `lane` of warp `warp` owns the KPL consecutive keys of a tile
        // that start at seg + lane * KPL: 128 bytes, eight 16-byte vectors.
        // It reads them in an order rotated by its lane -- register slot v
        // holds vector (v + lane) & 7 -- so that the eight lanes of each
        // quarter-warp read eight distinct bank groups; consecutive slots
        // hold consecutive vectors, except where the rotation wraps, at the
        // lane's first key.
        const int seg = warp * 32 * KPL;                      // the warp's first key in a tile
        const int rot = lane & 7;
        const uint32_t pos0 = (uint32_t)(seg + lane * KPL);   // the lane's first key in a tile
        // A dense tile waiting for the next iteration's pass: its stage, slot
        // and the slot's phase parity (pend_at: stage | slot << 8 | parity <<
        // 16), its tile (n < 2^32, so tile ids fit 32 bits), the pair of its
        // keys before this warp's, and the lane's head mask and heads of the
        // warp before its keys.
        uint32_t pend_at = 0, pend_tile = 0, pend_m = 0, pend_before = 0;
        bool pend = false;
        P pend_wex = 0;
        // Writes the pending dense tile once its pair is known, in rows of 32
        // lanes x EPL keys: per row the row's runs -- run indices [cw + first,
        // cw + first + nh) -- packed in this warp's slice of the stage, then
        // keys and lengths written with consecutive lanes on consecutive runs;
        // the warp hands the stage back after.  Lane l's chunk of row r lies
        // in the keys of lane 8r + l/4 in the pass, at bit EPL * (l % 4) of
        // its mask.
        auto write_dense = [&]() {
            const int ps = (int)(pend_at & 0xffu), pslot = (int)((pend_at >> 8) & 0xffu);
            const unsigned long long pbase = (unsigned long long)pend_tile * TILE;
            const bool pstaged = a.use_bulk && pbase + TILE <= n;
            if (!rle_wait(&prefix_ready[pslot], pend_at >> 16))
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
            if (warp == 0 && lane == 0) PS_TRACE_POINT(pend_tile, PS_TRACE_PREFIX_RECEIVED);
            const P pre = OpRle::combine(excl_of[pslot], pend_wex);
            const uint32_t cw = (uint32_t)(pre >> 32);
            const uint32_t wbase = (uint32_t)(pbase + (unsigned long long)seg);
            // the warp's keys again, in rows, all of them before the slice is reused
            KU kp[ROWS][EPL];
            if (pstaged) {
                const V *kv = reinterpret_cast<const V *>(stage_keys(ps));
                const int rr = (lane >> 2) & 1;   // pairs read in swapped order by lanes 4-7 of each quarter
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const int e0 = seg + (r * 32 + lane) * EPL;
                    const V x0 = kv[e0 / VK + rr], x1 = kv[e0 / VK + (rr ^ 1)];
                    const V lo = rr ? x1 : x0, hi = rr ? x0 : x1;
#pragma unroll
                    for (int j = 0; j < VK; ++j) {
                        kp[r][j] = KV::key(lo, j);
                        kp[r][VK + j] = KV::key(hi, j);
                    }
                }
            } else {
#pragma unroll
                for (int r = 0; r < ROWS; ++r)
#pragma unroll
                    for (int j = 0; j < EPL; ++j) {
                        const unsigned long long i = pbase + seg + (unsigned long long)((r * 32 + lane) * EPL + j);
                        kp[r][j] = i < n ? keys[i] : KU(0);
                    }
            }
            __syncwarp();
            KU *pk = stage_keys(ps) + seg;                                 // 32 * EPL keys
            uint32_t *pp = reinterpret_cast<uint32_t *>(pk + 32 * EPL);   // 32 * EPL offsets
            uint32_t row_prev = (uint32_t)pre;   // position of the last head before the row
            const uint32_t sh = (uint32_t)(EPL * (lane & 3));
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const int src = 8 * r + (lane >> 2);
                const uint32_t ml = __shfl_sync(kFull, pend_m, src);
                const uint32_t rb = __shfl_sync(kFull, pend_before, src) + (uint32_t)__popc(ml & ((1u << sh) - 1u));
                const uint32_t mr = (ml >> sh) & ((1u << EPL) - 1u);
                const uint32_t first = __shfl_sync(kFull, rb, 0);
                const uint32_t nh = __shfl_sync(kFull, rb + (uint32_t)__popc(mr), 31) - first;
                uint32_t q = rb - first;
#pragma unroll
                for (int j = 0; j < EPL; ++j)
                    if ((mr >> j) & 1u) {
                        pk[rle_sw(q)] = kp[r][j];
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
            // this warp is done with the stage
            if (lane == 0) {
                if (warp == 0) PS_TRACE_POINT(pend_tile, PS_TRACE_STORED);
                mbar_arrive(&empty[ps]);
            }
            pend = false;
        };
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            const int slot = (int)(k % R);
            if (!rle_wait(&full[s], (uint32_t)((k / S) & 1))) {
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
                    for (int i = 0; i < kLEnds; ++i) {
                        if (i > 0) tile_of[(k + i) % R] = num_tiles;
                        if (i < kLLB) mbar_arrive(&agg_done[(k + i) % R]);
                    }
                }
                __syncwarp();
                if (lane == 0)
#pragma unroll
                    for (int i = 0; i < kLW; ++i) mbar_arrive(&packed[(k + i) % R]);
                break;
            }
            const unsigned long long base = (unsigned long long)tile * TILE;
            const bool staged = a.use_bulk && base + TILE <= n;
            if (warp == 0 && lane == 0) {
                PS_TRACE_POINT(tile, PS_TRACE_DATA);
                PS_TRACE_POINT(tile, PS_TRACE_COMPUTE_START);
            }

            // Bit p of m: the lane's key p opens a run.
            const KU *ks = stage_keys(s);
            uint32_t m = 0;
            if (staged) {
                const V *kv = reinterpret_cast<const V *>(ks + pos0);
                KU kr[8][VK];
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const V x = kv[(v + rot) & 7];
#pragma unroll
                    for (int j = 0; j < VK; ++j) kr[v][j] = KV::key(x, j);
                }
                // in slot order, each key against the one in the slot before
                // (slot 0 against slot 7's last key: right except at the wrap)
                uint32_t mrot = 0;
#pragma unroll
                for (int v = 0; v < 8; ++v)
#pragma unroll
                    for (int j = 0; j < VK; ++j)
                        mrot |= (uint32_t)(kr[v][j] != (j ? kr[v][j - 1] : kr[(v + 7) & 7][VK - 1])) << (v * VK + j);
                m = rle_unrotate<KPL>(mrot, VK * rot);
                // bit 0 compared the lane's first key with its own last one;
                // the key before it is the previous lane's last (for lane 0 the
                // key before the warp, the tile's halo for warp 0)
                const KU first = pick_slot<KU, VK, 0>(kr, (8 - rot) & 7);
                const KU last = pick_slot<KU, VK, VK - 1>(kr, (7 - rot) & 7);
                KU prev = __shfl_up_sync(kFull, last, 1);
                if (lane == 0) prev = ks[seg - 1];
                m = (m & ~1u) | (uint32_t)(first != prev);
            } else {
#pragma unroll 4
                for (int p = 0; p < KPL; ++p) {
                    const unsigned long long i = base + pos0 + (unsigned long long)p;
                    m |= (uint32_t)(i < n && (i == 0 || keys[i] != keys[i - 1])) << p;
                }
            }
            if (tile == 0 && seg == 0 && lane == 0) m |= 1u;

            // the warp's heads before this lane's keys, its heads and its
            // last head (from the warp's first key)
            const uint32_t cnt = (uint32_t)__popc(m);
            const uint32_t sc = warp_inclusive<uint32_t>(cnt, lane);
            const uint32_t before = sc - cnt;
            const uint32_t run_c = __shfl_sync(kFull, sc, 31);
            const int run_last = __reduce_max_sync(kFull, m ? lane * KPL + 31 - __clz(m) : -1);
            P *sw = s_warp[k & 1];
            if (lane == 0)
                sw[warp] = ((P)run_c << 32) |
                           (run_last >= 0 ? (uint32_t)(base + (unsigned long long)(seg + run_last)) : 0u);
            named_barrier(1, CT);   // every warp has posted its pair
            if (aborted(&s_abort)) break;
            // the warps' pairs scanned across lanes 0 .. kLCW-1: the pair of
            // the tile's keys before this warp's, and the tile's
            P wp = lane < kLCW ? sw[lane] : (P)0;
#pragma unroll
            for (int d = 1; d < kLCW; d <<= 1) {
                const P o = __shfl_up_sync(kFull, wp, d);
                if (lane >= d) wp = OpRle::combine(o, wp);
            }
            const P agg = __shfl_sync(kFull, wp, kLCW - 1);
            P wex = __shfl_sync(kFull, wp, warp > 0 ? warp - 1 : 0);
            if (warp == 0) wex = 0;
            const bool sparse = (agg >> 32) <= (P)CAP;
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
                // writer is done with its previous tile: the keys come from
                // the stage, which goes back to the producer after
                const int o = (int)(k % NOB);
                if (k >= NOB && !rle_wait(&ob_empty[o], (uint32_t)((k / NOB - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    abort_meet(&s_abort, 1, CT);
                    break;
                }
                KU *ok = out_keys(o);
                uint16_t *op = out_pos(o);
                uint32_t q = (uint32_t)(wex >> 32) + before;
                for (uint32_t mm = m; mm; mm &= mm - 1u) {
                    const uint32_t p = pos0 + (uint32_t)(__ffs(mm) - 1);
                    ok[rle_sw(q)] = staged ? ks[p] : keys[base + p];
                    op[rle_sw(q)] = (uint16_t)p;
                    ++q;
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
                pend_m = m;
                pend_before = before;
            }
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
    long long grid = (long long)sms * kLCtasPerSm;
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
