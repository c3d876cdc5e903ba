// scan_persistent.cu -- the single-pass decoupled look-back scan as a
// persistent, TMA-fed kernel for sm_103a.
//
// One CTA per SM slot runs until the tiles run out.  Its warps split into
//   - CW compute warps, which scan tiles and store the results;
//   - one producer warp, whose elected lane takes the next tile id from the
//     global counter (dynamic tile ids: "virtual processors", section 4.4 of
//     the decoupled look-back paper summary; "Dynamic Block Index
//     Assignment" on the PMPP single-pass page) and copies the tile into a
//     ring of STAGES shared-memory buffers with one bulk asynchronous copy
//     (cp.async.bulk, completion counted in bytes on an mbarrier);
//   - one aggregator warp, which reduces each tile as soon as its copy has
//     landed and publishes the aggregate (A; P for tile 0) at once (step 3
//     of section 4.1), whatever the rest of the CTA is doing;
//   - one look-back warp, which then runs the warp-parallel look-back,
//     publishes P and hands the tile's exclusive prefix to the compute
//     warps (steps 4-5).
// The producer runs up to STAGES-1 tiles ahead, so the HBM reads of later
// tiles stay in flight, and the tile-id atomic leaves the critical path.
// Because a tile id is taken before its CTA is ready to scan it, publishing
// A only when some warp of the CTA gets round to it (after the scan, or
// after the previous tile's look-back) would make every successor wait for
// the slowest CTA; the aggregator publishes it when the data arrives.  The
// look-back usually finishes before the compute warps need the prefix, so
// its latency hides behind the scans of earlier tiles.
//
// Per tile the compute warps do steps a2-a5 and a9 as the one-tile-per-CTA
// kernel (scan_single_pass.cu) does: read the tile from shared memory in
// rows of 16-byte vectors (conflict-free) and hand the buffer straight back
// to the producer, scan in registers, combine warp totals, wait for the
// prefix, add it and store with 16-byte streaming stores.  Handing the
// buffer back before the prefix arrives keeps one more tile's read in
// flight per CTA; the per-iteration hand-offs between the roles therefore
// live in a ring of twice the stages (see kRing).
//
// A tile that is cut by the end of the array is not copied; the compute
// warps read it from global memory with bounds checks.  Every wait on an
// mbarrier is bounded; a wait that runs out records PS_ERR_LOOKBACK_TIMEOUT
// and the loop moves on (results are then unspecified, but the kernel ends).
#include <type_traits>

#include "scan_device.cuh"
#include "scan_pipeline.cuh"
#include "scan_trace.cuh"

namespace ps {

constexpr int kPCW = kThreads / 32;   // compute warps per CTA
// The compute warps hand a stage back as soon as they hold its data in
// registers (before the tile's prefix is known) unless this is 0; the
// per-iteration hand-offs then live in a ring of twice the stages.  A macro
// so that a tuning sweep can rebuild without it.
#ifndef PS_PERSIST_EARLY_RELEASE
#define PS_PERSIST_EARLY_RELEASE 1
#endif
constexpr bool kEarlyRelease = PS_PERSIST_EARLY_RELEASE != 0;
// At the start of a call thread 0 of each CTA prefetches into L2 the tiles
// the first round of claims will take, so their reads from memory overlap
// the header read and the tile-id atomics; 0 turns it off.
#ifndef PS_PERSIST_PREFETCH
#define PS_PERSIST_PREFETCH 1
#endif
// 16-byte vectors each compute lane holds per row for 8-byte elements: with
// two, a row's warp scan covers four elements per lane, as it does for 32-bit
// ones, so an int64 tile needs half the (two-shuffle) 64-bit warp scans.
#ifndef PS_PERSIST_VPL64
#define PS_PERSIST_VPL64 2
#endif
// The aggregator of an 8-byte commutative scan keeps one running value per
// vector element (two independent add-with-carry chains instead of one).
#ifndef PS_PERSIST_AGG_SPLIT64
#define PS_PERSIST_AGG_SPLIT64 1
#endif
// ... and of an fp32 scan one per vector element: four FADD chains of 64
// instead of one of 256 (the order of an fp32 tile sum is unspecified
// anyway; integer sums fold two additions per IADD3 already).
#ifndef PS_PERSIST_AGG_SPLIT_F32
#define PS_PERSIST_AGG_SPLIT_F32 1
#endif
// ... and of an int32 scan: four IADD chains of 64 rather than one chain
// of 128 IADD3s (data landed -> A published 0.96 -> 0.74 us at 2^26 with
// the unroll below).
#ifndef PS_PERSIST_AGG_SPLIT32
#define PS_PERSIST_AGG_SPLIT32 1
#endif
// Unroll of the aggregator's commutative loop for 4-byte and 8-byte
// elements (shared-memory loads in flight per lane).
#ifndef PS_PERSIST_AGG_UNROLL32
#define PS_PERSIST_AGG_UNROLL32 16
#endif
#ifndef PS_PERSIST_AGG_UNROLL64
#define PS_PERSIST_AGG_UNROLL64 8
#endif
constexpr int kRing = kEarlyRelease ? 2 * kPStages : kPStages;   // hand-off slots: iteration k uses k % kRing
// per stage: full, empty; per hand-off slot: agg_done, prefix_ready, tile id, aggregate, prefix
constexpr size_t kStageTailBytes = ((size_t)kPStages * 2 * 8 + (size_t)kRing * (2 * 8 + 8 + 8 + 8) + 127) / 128 * 128;

template <typename T> struct PItems { static constexpr int value = kItems32; };
template <> struct PItems<int64_t> { static constexpr int value = kItems64; };

template <typename T>
constexpr long long persistent_tile_elems() {
    return (long long)kPCW * 32 * PItems<T>::value;
}

template <typename T>
constexpr size_t persistent_smem_bytes() {
    // + per stage: 4 mbarriers, a tile id, an aggregate and a prefix
    return (size_t)kPStages * persistent_tile_elems<T>() * sizeof(T) + kStageTailBytes;
}

static_assert(kThreads % 32 == 0 && kThreads <= 960, "compute threads per CTA");


// LBW look-back warps per CTA; look-back warp j resolves the CTA's
// iterations j, j + LBW, ...  A second one lets a CTA resolve two tiles'
// prefixes at once: each look-back costs one or two L2 round trips of over a
// microsecond while the memory streams, close to the time in which a CTA
// moves a tile, so with one the tiles queue for it.  The launcher picks LBW
// from the array's length.
template <int LBW> constexpr int persistent_threads() { return (kPCW + 2 + LBW) * 32; }

template <typename T, bool EXCL, typename Op, int LBW>
__global__ void __launch_bounds__(persistent_threads<LBW>(), kPCtasPerSm)
persistent_kernel(PassArgs a, long long num_tiles) {
    static_assert(LBW >= 1 && LBW <= kPStages, "at most one look-back warp per stage");
    using Tr = Traits<T>;
    using U = typename Tr::U;
    const U ident = Op::template identity<U>();
    using V = typename Tr::V;
    constexpr int VEC = Tr::VEC;
    constexpr int ITEMS = PItems<T>::value;
    constexpr int VPL = sizeof(T) == 8 ? PS_PERSIST_VPL64 : 1;   // vectors per lane per row
    constexpr int EPL = VEC * VPL;                                // elements per lane per row
    constexpr int ROWS = ITEMS / EPL;
    static_assert(VPL == 1 || VPL == 2, "one or two vectors per lane per row");
    constexpr long long TILE = persistent_tile_elems<T>();
    constexpr uint32_t TILE_BYTES = (uint32_t)(TILE * sizeof(T));
    constexpr int CT = kPCW * 32;   // compute threads
    static_assert(ITEMS % EPL == 0, "ITEMS must be a multiple of a lane's share of a row");

    extern __shared__ __align__(128) unsigned char smem[];
    T *stage_data = reinterpret_cast<T *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kPStages * TILE_BYTES);
    __shared__ int s_abort;   // a compute warp's wait ran out: all of them leave
    uint64_t *empty = full + kPStages;
    uint64_t *agg_done = empty + kPStages;
    uint64_t *prefix_ready = agg_done + kRing;
    long long *tile_of = reinterpret_cast<long long *>(prefix_ready + kRing);
    U *agg_of = reinterpret_cast<U *>(tile_of + kRing);
    U *excl_of = agg_of + kRing;
    __shared__ U s_warp[2][kPCW];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    Header *hdr = reinterpret_cast<Header *>(a.ws);
    void *desc = a.ws + kHeaderBytes;
    const unsigned long long n = a.n;
    const T *in = reinterpret_cast<const T *>(a.in);
    T *out = reinterpret_cast<T *>(a.out);

    // Thread 0 alone reads the header and hands the verdict to the CTA: one
    // request per CTA to that L2 line, not one per warp (with 304 CTAs of 11
    // warps the per-warp reads queued for microseconds at the line's slice).
    __shared__ uint32_t s_epoch;
    __shared__ int s_ok;
    if (tid == 0) {
        PS_TRACE_CTA_POINT(PS_TRACE_CTA_ENTRY);
        if (PS_PERSIST_PREFETCH) {
            // The producers take up to kPStages tile ids each before any
            // stage comes back, so the first claims fall on the first
            // kPStages x gridDim.x tiles, in whatever order: CTA b warms
            // tiles b, b + grid and b + 2 grid (those the bulk copy will
            // read).  Each is bulk-loaded soon after, so this adds no traffic.
            for (int j = 0; j < kPStages; ++j) {
                const unsigned long long t = blockIdx.x + (unsigned long long)j * gridDim.x;
                if ((t + 1) * (unsigned long long)TILE <= n) prefetch_l2(in + t * TILE, TILE_BYTES);
            }
        }
        uint32_t e;
        s_ok = begin_call(hdr, &e) ? 1 : 0;
        s_epoch = e;
        s_abort = 0;
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPCW + 1);     // compute warps + aggregator
        }
        for (int slot = 0; slot < kRing; ++slot) {
            mbar_init(&agg_done[slot], 1);
            mbar_init(&prefix_ready[slot], 1);
            tile_of[slot] = num_tiles;   // end marker until the producer fills it
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!s_ok) return;   // same verdict in every CTA: nothing runs
    const uint32_t epoch = s_epoch;
    if (tid == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_HEADER);

    if (warp == kPCW) {
        // ---------------- producer warp ----------------
        if (lane == 0) {
            for (long long k = 0;; ++k) {
                const int s = (int)(k % kPStages);
                if (k >= kPStages) {
                    const uint32_t parity = (uint32_t)((k / kPStages - 1) & 1);
                    if (!mbar_wait(&empty[s], parity)) {   // never in a correct run
                        report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                        break;
                    }
                }
                const long long t = (long long)atomicAdd(&hdr->tile_counter, 1ull);
                if (t < num_tiles) {
                    PS_TRACE_POINT(t, PS_TRACE_CLAIM);
                    PS_TRACE_CTA(t);
                }
                tile_of[k % kRing] = t;
                if (t < num_tiles) prefetch_descriptor<Tr::DW>(desc, t);
                if (t < num_tiles && (unsigned long long)(t + 1) * TILE <= n) {
                    mbar_arrive_expect_tx(&full[s], TILE_BYTES);
                    bulk_load(stage_data + (size_t)s * TILE, in + t * TILE, TILE_BYTES, &full[s]);
                } else {
                    mbar_arrive(&full[s]);   // end marker, or a cut tile read from global
                }
                if (t >= num_tiles) break;
            }
            if (epoch != kEpochMask) claims_done(hdr, a.ws_bytes, epoch);
        }
    } else if (warp == kPCW + 1) {
        // ---------------- aggregator warp ----------------
        // Reduces each tile as soon as its copy lands and publishes A (P for
        // tile 0) at once, independently of any look-back (step 3 of
        // section 4.1).
        for (long long k = 0;; ++k) {
            const int s = (int)(k % kPStages);
            if (!mbar_wait(&full[s], (uint32_t)((k / kPStages) & 1))) {   // never in a correct run
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const int slot = (int)(k % kRing);
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) {
                // end marker: pass it on to every look-back warp, on the
                // slots of the next LBW iterations (the producer, which
                // stopped here, writes none of them again)
                if (lane == 0) {
#pragma unroll
                    for (int i = 0; i < LBW; ++i) {
                        if (i > 0) tile_of[(k + i) % kRing] = num_tiles;
                        mbar_arrive(&agg_done[(k + i) % kRing]);
                    }
                }
                break;
            }
            const unsigned long long tile_base = (unsigned long long)tile * TILE;
            if (lane == 0) PS_TRACE_POINT(tile, PS_TRACE_DATA);
            U agg;
            if constexpr (Op::kCommutative) {
                // each lane folds every 32nd vector; the order does not matter
                constexpr int AC = (sizeof(U) == 8 && PS_PERSIST_AGG_SPLIT64) ? VEC
                                   : (std::is_same<U, float>::value && PS_PERSIST_AGG_SPLIT_F32) ? VEC
                                   : (std::is_same<U, uint32_t>::value && PS_PERSIST_AGG_SPLIT32) ? VEC : 1;
                constexpr int UNROLL = sizeof(U) == 8 ? PS_PERSIST_AGG_UNROLL64 : PS_PERSIST_AGG_UNROLL32;
                U accs[AC];
#pragma unroll
                for (int c = 0; c < AC; ++c) accs[c] = ident;
                if (tile_base + TILE <= n) {
                    const V *src = reinterpret_cast<const V *>(stage_data + (size_t)s * TILE);
#pragma unroll UNROLL
                    for (int i = lane; i < (int)(TILE / VEC); i += 32) {
                        const V x = src[i];
#pragma unroll
                        for (int j = 0; j < VEC; ++j) accs[j % AC] = Op::combine(accs[j % AC], (U)vget(x, j));
                    }
                } else {
                    for (unsigned long long i = tile_base + lane; i < n; i += 32) accs[0] = Op::combine(accs[0], (U)in[i]);
                }
                U acc = accs[0];
#pragma unroll
                for (int c = 1; c < AC; ++c) acc = Op::combine(acc, accs[c]);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                agg = warp_reduce<U, Op>(acc);
            } else {
                // in sequence order: lane l folds the l-th 32nd of the tile,
                // C consecutive vectors, then the lanes' partials are folded
                // towards lane 0, earlier on the left.  Lane l visits its
                // vectors starting at r = l mod 8, so that the 8 lanes one
                // 16-byte shared-memory load serves hit distinct banks: it
                // folds [r, C) and [0, r) separately and joins them in order.
                U running = ident;
                if (tile_base + TILE <= n) {
                    constexpr int C = (int)(TILE / VEC / 32);
                    static_assert(C >= 8 && (C & (C - 1)) == 0, "chunk of a power-of-two size >= 8");
                    const V *src = reinterpret_cast<const V *>(stage_data + (size_t)s * TILE) + lane * C;
                    const int r = lane & 7;
                    U tail = ident, head = ident;
#pragma unroll 4
                    for (int q = 0; q < C; ++q) {
                        const int vi = (q + r) & (C - 1);
                        const V x = src[vi];
                        U p = (U)vget(x, 0);
#pragma unroll
                        for (int j = 1; j < VEC; ++j) p = Op::combine(p, (U)vget(x, j));
                        if (vi >= r) tail = Op::combine(tail, p);
                        else head = Op::combine(head, p);
                    }
                    U p = Op::combine(head, tail);
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const U o = __shfl_down_sync(kFull, p, d);
                        if (lane + d < 32) p = Op::combine(p, o);
                    }
                    running = __shfl_sync(kFull, p, 0);
                } else {
                    for (unsigned long long i0 = tile_base; i0 < n; i0 += 32) {
                        const unsigned long long i = i0 + lane;
                        U p = i < n ? (U)in[i] : ident;
#pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {
                            const U o = __shfl_down_sync(kFull, p, d);
                            if (lane + d < 32) p = Op::combine(p, o);
                        }
                        running = Op::combine(running, __shfl_sync(kFull, p, 0));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                agg = running;
            }
            if (lane == 0) {
                if (tile == 0) {
                    // the only read of carry_in: it precedes tile 0's P, hence
                    // every other tile's P and the write of carry_out, so
                    // carry_in may alias carry_out
                    const U c = a.carry_in ? *reinterpret_cast<const U *>(a.carry_in) : ident;
                    Desc<U, Tr::DW>::store(desc, 0, kFlagP, Op::combine(c, agg), epoch);
                    excl_of[slot] = c;   // for the look-back warp
                } else {
                    Desc<U, Tr::DW>::store(desc, tile, kFlagA, agg, epoch);
                }
                agg_of[slot] = agg;
                PS_TRACE_POINT(tile, PS_TRACE_AGGREGATE);
                mbar_arrive(&agg_done[slot]);
            }
        }
    } else if (warp == kPCW + 2 || (LBW > 1 && warp > kPCW + 2)) {
        // ---------------- look-back warps ----------------
        // Run ahead of the compute warps: once a tile's A is out its
        // look-back warp looks back, publishes P and leaves the exclusive
        // prefix in excl_of[slot] (steps 4-5 of section 4.1), so the compute
        // warps rarely wait.
        // Warp j takes iterations j, j + LBW, ...; the slot and the phase
        // parity are stepped directly (LBW divides the ring), which keeps
        // 64-bit divisions out of the loop and the kernel within its
        // register budget.
        static_assert(kRing % LBW == 0, "the look-back warps step through the ring evenly");
        int slot = LBW == 1 ? 0 : warp - (kPCW + 2);
        uint32_t parity = 0;
        for (;; slot += LBW) {
            if (slot >= kRing) {
                slot -= kRing;
                parity ^= 1u;
            }
            if (!mbar_wait(&agg_done[slot], parity)) {   // never in a correct run
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            const U agg = agg_of[slot];
            if (lane == 0) PS_TRACE_POINT(tile, PS_TRACE_LOOKBACK_START);
            __syncwarp();
            U excl;
            if (tile == 0) {
                excl = excl_of[slot];   // the carry the aggregator read
            } else {
                excl = look_back<U, Tr::DW, kLookbackK, Op>(desc, tile, epoch, a.max_polls, &hdr->status,
                                                            PS_TRACE_LOOKBACK(tile));
                if (lane == 0) Desc<U, Tr::DW>::store(desc, tile, kFlagP, Op::combine(excl, agg), epoch);
            }
            if (lane == 0) {
                if (a.carry_out && tile == num_tiles - 1) *reinterpret_cast<U *>(a.carry_out) = Op::combine(excl, agg);
                excl_of[slot] = excl;
                PS_TRACE_POINT(tile, PS_TRACE_PREFIX);
                mbar_arrive(&prefix_ready[slot]);
            }
        }
    } else {
    // ---------------- compute warps ----------------
    for (long long k = 0;; ++k) {
        const int s = (int)(k % kPStages);
        if (!mbar_wait(&full[s], (uint32_t)((k / kPStages) & 1))) {   // never in a correct run
            report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
            abort_meet(&s_abort, 1, CT);
            break;
        }
        const int slot = (int)(k % kRing);
        const long long tile = tile_of[slot];
        if (tile < 0 || tile >= num_tiles) break;
        const unsigned long long tile_base = (unsigned long long)tile * TILE;
        const bool cut = tile_base + TILE > n;
        const int seg = warp * 32 * ITEMS;   // element offset of this warp in the tile
        if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_COMPUTE_START);

        // a2: rows of 16-byte vectors from the stage (or bounded global loads)
        // With two vectors per lane, lanes 4-7 of each quarter-warp read
        // their pair in swapped order, so that the eight 16-byte reads of a
        // quarter-warp fall in distinct bank groups; the pair is put back in
        // order in registers.
        U v[ROWS][EPL];
        if (!cut) {
            const V *src = reinterpret_cast<const V *>(stage_data + (size_t)s * TILE + seg) + lane * VPL;
            const int rot = VPL == 2 ? (lane >> 2) & 1 : 0;
            V buf[ROWS][VPL];
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int t = 0; t < VPL; ++t) buf[r][t] = src[r * 32 * VPL + (t ^ rot)];
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int t = 0; t < VPL; ++t) {
                    const V x = rot ? buf[r][t ^ 1] : buf[r][t];
#pragma unroll
                    for (int j = 0; j < VEC; ++j) v[r][t * VEC + j] = (U)vget(x, j);
                }
            if (kEarlyRelease) {
                // the tile is in registers: the stage goes back to the
                // producer before the prefix arrives.  The producer stays
                // within kPStages iterations of this release and the compute
                // warps within one of the look-back warp, so a hand-off slot
                // (and its mbarrier phase) is not reused while a reader still
                // needs it.
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
        } else {
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const unsigned long long i = tile_base + seg + (unsigned long long)(r * 32 + lane) * EPL + j;
                    v[r][j] = i < n ? (U)in[i] : ident;
                }
        }
        // a3 + a4.  For 8-byte inclusive scans each row's offset within the warp
        // is folded into its values at once rather than kept until the
        // prefix arrives: ROWS more live 64-bit words would push the
        // compute warps past the 80 registers that two CTAs of this size
        // per SM allow (the cap is per SM sub-partition), and they spilled.
        constexpr bool kFoldRows = sizeof(U) == 8 && !EXCL;
        U off[kFoldRows ? 1 : ROWS];
        U running = ident;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            U t;
            if (EXCL) {
                U acc = ident;
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const U x = v[r][j];
                    v[r][j] = acc;
                    acc = Op::combine(acc, x);
                }
                t = acc;
            } else {
#pragma unroll
                for (int j = 1; j < EPL; ++j) v[r][j] = Op::combine(v[r][j - 1], v[r][j]);
                t = v[r][EPL - 1];
            }
            const U sc = warp_inclusive<U, Op>(t, lane);
            U le = __shfl_up_sync(kFull, sc, 1);
            if (lane == 0) le = ident;
            const U row_total = __shfl_sync(kFull, sc, 31);
            if constexpr (kFoldRows) {
                const U o = Op::combine(running, le);
#pragma unroll
                for (int j = 0; j < EPL; ++j) v[r][j] = Op::combine(o, v[r][j]);
            } else {
                off[r] = Op::combine(running, le);
            }
            running = Op::combine(running, row_total);
        }

        // a5 (double-buffered by iteration, so that no second barrier is needed)
        U *sw = s_warp[k & 1];
        if (lane == 0) sw[warp] = running;
        named_barrier(1, CT);
        if (aborted(&s_abort)) break;
        U warp_excl = ident;
#pragma unroll
        for (int w = 0; w < kPCW; ++w)
            if (w < warp) warp_excl = Op::combine(warp_excl, sw[w]);

        // the look-back warp provides the tile's exclusive prefix
        if (!mbar_wait(&prefix_ready[slot], (uint32_t)((k / kRing) & 1)))   // never in a correct run
            report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
        const U tile_excl = excl_of[slot];
        if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_PREFIX_RECEIVED);

        // a9
        const U base = Op::combine(tile_excl, warp_excl);
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const U o = kFoldRows ? base : Op::combine(base, off[r]);
#pragma unroll
            for (int j = 0; j < EPL; ++j) v[r][j] = Op::combine(o, v[r][j]);
        }
        if (!cut) {
            if constexpr (VPL == 2) {
                // a lane's 32 bytes of a row in one store when `out` allows it
                // (the bulk-copy path needs only 16-byte alignment)
                V *dst = reinterpret_cast<V *>(out + tile_base + seg) + lane * 2;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    V w0, w1;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        vset(w0, j, v[r][j]);
                        vset(w1, j, v[r][VEC + j]);
                    }
                    if ((reinterpret_cast<uintptr_t>(out) & 31) == 0) {
                        st_stream_pair(dst + r * 64, w0, w1);
                    } else {
                        st_stream(dst + r * 64, w0);
                        st_stream(dst + r * 64 + 1, w1);
                    }
                }
            } else {
                V *dst = reinterpret_cast<V *>(out + tile_base + seg) + lane;
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    V w;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) vset(w, j, v[r][j]);
                    st_stream(dst + r * 32, w);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const unsigned long long i = tile_base + seg + (unsigned long long)(r * 32 + lane) * EPL + j;
                    if (i < n) out[i] = (T)v[r][j];
                }
        }
        // Without the early release (or for a cut tile, read from global)
        // the stage goes back only now; the look-back warp then cannot run a
        // whole ring ahead on it, so each hand-off phase completes once per
        // use and the parity wait above cannot alias.
        if (!kEarlyRelease || cut) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_STORED);
    }
    if (warp == 0 && lane == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_DONE);
    }

    // The last producer to take its last tile id readied the workspace
    // (claims_done); before an epoch wrap the last CTA to finish does.
    if (epoch == kEpochMask) finish_call(hdr, a.ws, a.ws_bytes, epoch);
}

// Two look-back warps per CTA for arrays of [FROM, BELOW) tiles per CTA slot
// of a full grid, one otherwise.  Macros so that a sweep can rebuild with
// other bounds.
#ifndef PS_PERSIST_LBW2_FROM
#define PS_PERSIST_LBW2_FROM 0
#endif
#ifndef PS_PERSIST_LBW2_BELOW
#define PS_PERSIST_LBW2_BELOW 12
#endif

// Internal linkage (static) for the launchers that keep a function-local
// static: an external template instance's local static is a process-wide
// (GNU-unique) symbol, so a second copy of this library loaded into the same
// process would share the first one's record and skip its own opt-in.
template <typename T, bool EXCL, typename Op, int LBW>
static cudaError_t launch_persistent_lbw(const PassArgs &a, long long tiles, int dev, long long grid, cudaStream_t s) {
    constexpr size_t smem = persistent_smem_bytes<T>();
    // the dynamic shared-memory opt-in, once per device and template instance
    // (a repeated call from a racing thread is harmless)
    static volatile int configured[64] = {};
    cudaError_t e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(persistent_kernel<T, EXCL, Op, LBW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    persistent_kernel<T, EXCL, Op, LBW><<<(unsigned int)grid, persistent_threads<LBW>(), smem, s>>>(a, tiles);
    return cudaGetLastError();
}

template <typename T, bool EXCL, typename Op>
static cudaError_t launch_persistent_kind(const PassArgs &a, cudaStream_t s) {
    const long long tiles = (long long)((a.n + persistent_tile_elems<T>() - 1) / persistent_tile_elems<T>());
    cudaError_t e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const long long full = (long long)sms * kPCtasPerSm;
    const long long grid = full < tiles ? full : tiles;
    if (tiles >= (long long)PS_PERSIST_LBW2_FROM * full && tiles < (long long)PS_PERSIST_LBW2_BELOW * full)
        return launch_persistent_lbw<T, EXCL, Op, 2>(a, tiles, dev, grid, s);
    return launch_persistent_lbw<T, EXCL, Op, 1>(a, tiles, dev, grid, s);
}

template <typename T, typename Op>
static cudaError_t launch_persistent_op(const PassArgs &a, bool exclusive, cudaStream_t s) {
    return exclusive ? launch_persistent_kind<T, true, Op>(a, s) : launch_persistent_kind<T, false, Op>(a, s);
}

template <typename T>
cudaError_t launch_persistent(const PassArgs &a, bool exclusive, int op, cudaStream_t s) {
    if constexpr (sizeof(T) == 8) {   // the pair element types travel as int64 words
        if (op == kOpPairI32F32) return launch_persistent_op<T, OpPairI32F32>(a, exclusive, s);
        if (op == kOpAffineF32) return launch_persistent_op<T, OpAffineF32>(a, exclusive, s);
    }
    switch (op) {
    case kOpMax: return launch_persistent_op<T, OpMax>(a, exclusive, s);
    case kOpMin: return launch_persistent_op<T, OpMin>(a, exclusive, s);
    default: return launch_persistent_op<T, OpSum>(a, exclusive, s);
    }
}

template cudaError_t launch_persistent<int32_t>(const PassArgs &, bool, int, cudaStream_t);
template cudaError_t launch_persistent<int64_t>(const PassArgs &, bool, int, cudaStream_t);
template cudaError_t launch_persistent<float>(const PassArgs &, bool, int, cudaStream_t);

}  // namespace ps

namespace ps {
TRACE_COPY_FUNCTIONS(trace_copy_scan, trace_copy_scan_ctas)
}  // namespace ps
