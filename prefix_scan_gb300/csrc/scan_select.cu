// scan_select.cu -- single-pass stream compaction: select and partition.
//
// The output position of a kept element is the exclusive prefix sum of the
// 0/1 selection flags (decoupled look-back paper summary, section 4.4,
// "in-place compaction behaviour"), so compaction is the single-pass scan of
// the flags with a scatter fused into its last step:
//   select     out[count of selected before i] = x[i] for every selected i;
//   partition  the same for selected elements, and every other element i
//              goes to out[n - 1 - (i - count of selected before i)], i.e.
//              the rejected ones fill the array from the back in reverse
//              order -- a position known without the final count.
// Selection is a flag array (nonzero = keep) or a predicate on the value
// (nonzero, greater than a threshold, less than a threshold).
//
// Same structure as the persistent scan kernel (scan_persistent.cu): a
// producer warp takes tile ids and bulk-copies values (and flags) into a
// shared-memory ring, an aggregator warp counts each tile's selected
// elements and publishes the count at once, a look-back warp resolves the
// tile's offset, and the compute warps scan the flags in registers and
// scatter.  Counts are 32-bit (n < 2^32).
//
// In place (out == in, select only) is safe because a tile learns its
// offset only after every predecessor has published its count, which each
// does after its data sits in shared memory: nothing is overwritten that a
// predecessor still has to read, and a tile never writes past its own end.
// That argument needs the bulk copies, so in place requires 16-byte
// aligned values and flags.
#include "scan_device.cuh"
#include "scan_cluster.cuh"
#include "scan_pipeline.cuh"
#include "scan_trace.cuh"

namespace ps {

namespace {

// Compute warps per CTA and CTAs per SM (macros, so that a tuning sweep can
// rebuild).
#ifndef PS_SEL_COMPUTE_WARPS
#define PS_SEL_COMPUTE_WARPS (PS_THREADS / 32)
#endif
#ifndef PS_SEL_CTAS_PER_SM
#define PS_SEL_CTAS_PER_SM PS_PERSIST_CTAS_PER_SM
#endif
constexpr int kSCW = PS_SEL_COMPUTE_WARPS;
constexpr int kSCtasPerSm = PS_SEL_CTAS_PER_SM;

// Elements per thread of a select / partition tile and the stages of the
// flag-array form (macros so that a tuning sweep can rebuild with others).
#ifndef PS_SEL_ITEMS32
#define PS_SEL_ITEMS32 PS_ITEMS32
#endif
#ifndef PS_SEL_FLAG_STAGES
#define PS_SEL_FLAG_STAGES 2
#endif
// Look-back warps per CTA; warp j resolves iterations j, j + LB, ...  Two
// for partition, whose 2 stages plus pack buffer hold each tile longer, so
// that a CTA has two look-backs in flight: at 2^28, 436.6 -> 425.2 us; one
// for select, which a second made slower (310.6 -> 319.1 us).  Macros so
// that a tuning sweep can rebuild.
#ifndef PS_SEL_LOOKBACK_WARPS
#define PS_SEL_LOOKBACK_WARPS 1
#endif
#ifndef PS_PART_LOOKBACK_WARPS
#define PS_PART_LOOKBACK_WARPS 2
#endif
template <bool PARTITION> constexpr int sel_lookback_warps() {
    return PARTITION ? PS_PART_LOOKBACK_WARPS : PS_SEL_LOOKBACK_WARPS;
}
// compute, producer, aggregator and look-back warps
template <bool PARTITION> constexpr int sel_threads() { return (kSCW + 2 + sel_lookback_warps<PARTITION>()) * 32; }
template <typename T> struct SelItems { static constexpr int value = PS_SEL_ITEMS32; };
template <> struct SelItems<int64_t> { static constexpr int value = kItems64; };

template <typename T> constexpr long long sel_tile() { return (long long)kSCW * 32 * SelItems<T>::value; }
// Stages: 2 with a flag array (values + flags, 40 KiB per int32 tile), else
// 3; partition keeps 2 either way to make room for its pack buffer.
template <int OP, bool PARTITION> constexpr int sel_stages() {
    return OP == 0 ? PS_SEL_FLAG_STAGES : PARTITION ? 2 : kPStages;
}
template <typename T, int OP> constexpr size_t sel_stage_bytes() {
    return (size_t)sel_tile<T>() * sizeof(T) + (OP == 0 ? (size_t)sel_tile<T>() : 0);
}
// Per-iteration hand-offs (tile id, count, offset and their two mbarriers)
// live in a ring of twice as many slots as there are stages, so that a
// stage can be handed back before its offset has been consumed (select).
template <int OP, bool PARTITION> constexpr int sel_ring() { return 2 * sel_stages<OP, PARTITION>(); }
// partition: one tile of values in which each warp packs its output
template <typename T, bool PARTITION> constexpr size_t sel_pack_bytes() {
    return PARTITION ? (size_t)sel_tile<T>() * sizeof(T) : 0;
}
template <typename T, int OP, bool PARTITION> constexpr size_t sel_smem_bytes() {
    return (size_t)sel_stages<OP, PARTITION>() * sel_stage_bytes<T, OP>() + sel_pack_bytes<T, PARTITION>() +
           ((size_t)sel_stages<OP, PARTITION>() * 2 * 8 + (size_t)sel_ring<OP, PARTITION>() * (2 * 8 + 8 + 4 + 4) +
            127) / 128 * 128;
}

// Raw bits of the element type, for comparisons in the element's own type.
template <typename T> __device__ __forceinline__ T from_raw(unsigned long long b);
template <> __device__ __forceinline__ int32_t from_raw<int32_t>(unsigned long long b) { return (int32_t)(uint32_t)b; }
template <> __device__ __forceinline__ int64_t from_raw<int64_t>(unsigned long long b) { return (int64_t)b; }
template <> __device__ __forceinline__ float from_raw<float>(unsigned long long b) { return __uint_as_float((uint32_t)b); }

// OP: 0 flag array, 1 nonzero, 2 greater than t, 3 less than t
template <typename T, int OP>
__device__ __forceinline__ bool keep(T x, uint8_t f, T t) {
    if (OP == 0) return f != 0;
    if (OP == 1) return x != T(0);
    if (OP == 2) return x > t;
    return x < t;
}

template <typename T> __device__ __forceinline__ T vget_t(const typename Traits<T>::V &v, int j);
template <> __device__ __forceinline__ int32_t vget_t<int32_t>(const uint4 &v, int j) { return (int32_t)vget(v, j); }
template <> __device__ __forceinline__ float vget_t<float>(const float4 &v, int j) { return vget(v, j); }
template <> __device__ __forceinline__ int64_t vget_t<int64_t>(const ulonglong2 &v, int j) { return (int64_t)vget(v, j); }

// The lane's part of a tile's kept count (the aggregator warp sums the
// lanes'): from the stage when the tile was bulk-copied, else from global
// memory with bounds (a tile cut by the end of the array, or past it).
template <typename T, int OP>
__device__ __forceinline__ uint32_t count_tile(const SelectArgs &a, T thr, const T *vals_s, const uint8_t *flg_s,
                                               unsigned long long base, int lane) {
    using V = typename Traits<T>::V;
    constexpr int VEC = Traits<T>::VEC;
    constexpr long long TILE = sel_tile<T>();
    const unsigned long long n = a.n;
    const T *in = reinterpret_cast<const T *>(a.in);
    uint32_t cnt = 0;
    if (a.use_bulk && base + TILE <= n) {
        if (OP == 0) {
            // __vcmpne4 sets a byte to 0xff where the flag byte is nonzero:
            // eight set bits per kept element
            const uint4 *f4 = reinterpret_cast<const uint4 *>(flg_s);
            uint32_t bits = 0;
#pragma unroll 4
            for (int i = lane; i < (int)(TILE / 16); i += 32) {
                const uint4 w = f4[i];
                bits += __popc(__vcmpne4(w.x, 0u)) + __popc(__vcmpne4(w.y, 0u)) +
                        __popc(__vcmpne4(w.z, 0u)) + __popc(__vcmpne4(w.w, 0u));
            }
            cnt = bits >> 3;
        } else {
            const V *src = reinterpret_cast<const V *>(vals_s);
            for (int i = lane; i < (int)(TILE / VEC); i += 32) {
                const V x = src[i];
#pragma unroll
                for (int j = 0; j < VEC; ++j) cnt += keep<T, OP>(vget_t<T>(x, j), 0, thr);
            }
        }
    } else {
        const unsigned long long end = base + TILE < n ? base + TILE : n;
        for (unsigned long long i = base + lane; i < end; i += 32)
            cnt += keep<T, OP>(OP == 0 ? T(0) : in[i], OP == 0 ? a.flags[i] : (uint8_t)0, thr);
    }
    return cnt;
}

// One tile's pass by the compute warps: the values (and flags) into
// registers, the stage back to the producer (it is not read again), the
// kept elements counted within each warp and across the warps, then -- once
// wait_prefix() has the tile's output offset -- the scatter.  Select writes
// each warp row's kept elements, one contiguous run, straight from the
// registers; partition packs each warp's kept elements and then its
// rejected ones into the warp's slice of the pack buffer and writes them as
// two contiguous runs (the rejected one downwards from the end of `out`).
// False when the compute warps' abort flag is up (a wait ran out).
template <typename T, int OP, bool PARTITION, typename WaitPrefix>
__device__ __forceinline__ bool select_tile_pass(const SelectArgs &a, T thr, long long tile, const T *vals_s,
                                                 const uint8_t *flg_s, T *pack, uint64_t *empty_s, uint32_t *sw,
                                                 volatile int *abort_flag, WaitPrefix wait_prefix) {
    using V = typename Traits<T>::V;
    using U = uint32_t;
    constexpr int VEC = Traits<T>::VEC;
    constexpr int ITEMS = SelItems<T>::value;
    constexpr int ROWS = ITEMS / VEC;
    constexpr long long TILE = sel_tile<T>();
    constexpr int CT = kSCW * 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned long long n = a.n;
    const T *in = reinterpret_cast<const T *>(a.in);
    T *out = reinterpret_cast<T *>(a.out);
    const unsigned long long base = (unsigned long long)tile * TILE;
    const bool staged = a.use_bulk && base + TILE <= n;
    const int seg = warp * 32 * ITEMS;
    if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_COMPUTE_START);

    T v[ROWS][VEC];
    uint32_t sel[ROWS];   // bit j: element j of this lane's row chunk is kept
    if (staged) {
        const V *src = reinterpret_cast<const V *>(vals_s + seg) + lane;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const V x = src[r * 32];
            uint32_t fb = 0;
            if (OP == 0) {
                const uint8_t *fp = flg_s + seg + (r * 32 + lane) * VEC;
                fb = VEC == 4 ? *reinterpret_cast<const uint32_t *>(fp)
                              : (uint32_t)*reinterpret_cast<const uint16_t *>(fp);
            }
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                v[r][j] = vget_t<T>(x, j);
                m |= (uint32_t)keep<T, OP>(v[r][j], (uint8_t)(fb >> (8 * j)), thr) << j;
            }
            sel[r] = m;
        }
    } else {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const unsigned long long i = base + seg + (unsigned long long)(r * 32 + lane) * VEC + j;
                v[r][j] = i < n ? in[i] : T(0);
                const bool kp = i < n && keep<T, OP>(v[r][j], OP == 0 ? a.flags[i] : (uint8_t)0, thr);
                m |= (uint32_t)kp << j;
            }
            sel[r] = m;
        }
    }

    // the tile is in registers and the stage is not read again: it goes
    // back to the producer now, before the offset arrives (the hand-off ring
    // keeps the slots apart)
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_s);
    // exclusive count of kept elements before each lane's row chunk
    U off[ROWS];
    U running = 0;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const U t = (U)__popc(sel[r]);
        const U sc = warp_inclusive<U>(t, lane);
        off[r] = running + (sc - t);
        running += __shfl_sync(kFull, sc, 31);
    }
    if (lane == 0) sw[warp] = running;
    named_barrier(1, CT);
    if (aborted(abort_flag)) return false;
    U warp_excl = 0;
#pragma unroll
    for (int w = 0; w < kSCW; ++w)
        if (w < warp) warp_excl += sw[w];
    const U tile_excl = wait_prefix();
    if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_PREFIX_RECEIVED);

    if (!PARTITION) {
        // select: kept elements straight to their places; within a warp row
        // they form one contiguous run
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const U before = tile_excl + warp_excl + off[r];
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if ((sel[r] >> j) & 1u) out[before + (U)__popc(sel[r] & ((1u << j) - 1u))] = v[r][j];
        }
    } else {
        // partition: each warp packs its kept elements, then its rejected
        // ones, into its own slice of the pack buffer and writes them as two
        // contiguous runs, consecutive lanes to consecutive addresses
        T *wbuf = pack + seg;
        const U w_sel = running;   // kept elements of this warp
        const unsigned long long w_first = base + seg;
        const U w_valid = w_first >= n ? 0u
                          : (n - w_first >= (unsigned long long)(32 * ITEMS) ? (U)(32 * ITEMS)
                                                                            : (U)(n - w_first));
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            // c: kept elements of the warp before element e (a running count
            // over the chunk); a rejected element goes after the warp's kept
            // ones, at its count of rejected predecessors
            U c = off[r];
            const U e0 = (U)((r * 32 + lane) * VEC);   // index within the warp's slice
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                const U e = e0 + (U)j;
                const bool kp = (sel[r] >> j) & 1u;
                const U pos = kp ? c : w_sel + (e - c);
                if (kp || e < w_valid) wbuf[pos] = v[r][j];
                c += kp ? 1u : 0u;
            }
        }
        __syncwarp();
        const U dst = tile_excl + warp_excl;   // kept elements before this warp
        for (U q = lane; q < w_sel; q += 32) out[dst + q] = wbuf[q];
        const unsigned long long rej_before = w_first - dst;   // rejected before this warp
        const U w_rej = w_valid - w_sel;
        for (U q = lane; q < w_rej; q += 32) out[n - 1 - (rej_before + q)] = wbuf[w_sel + q];
        __syncwarp();   // the slice is packed again next iteration
    }
    if (warp == 0 && lane == 0) PS_TRACE_POINT(tile, PS_TRACE_STORED);
    return true;
}

}  // namespace


template <typename T, int OP, bool PARTITION>
__global__ void __launch_bounds__(sel_threads<PARTITION>(), kSCtasPerSm)
select_kernel(SelectArgs a, long long num_tiles) {
    using U = uint32_t;                     // counts
    constexpr int VEC = Traits<T>::VEC;
    constexpr int ITEMS = SelItems<T>::value;
    constexpr long long TILE = sel_tile<T>();
    constexpr int S = sel_stages<OP, PARTITION>();
    constexpr int R = sel_ring<OP, PARTITION>();
    constexpr uint32_t VAL_BYTES = (uint32_t)(TILE * sizeof(T));
    constexpr uint32_t FLAG_BYTES = OP == 0 ? (uint32_t)TILE : 0u;
    constexpr int CT = kSCW * 32;
    constexpr int LB = sel_lookback_warps<PARTITION>();
    static_assert(ITEMS % VEC == 0, "ITEMS must be a multiple of the vector width");
    // the producer sends one end marker per look-back warp, each in a stage
    // of its own, and the compute warps hand back none after the first
    static_assert(LB <= S, "at most one look-back warp per stage");

    extern __shared__ __align__(128) unsigned char smem[];
    T *vals = reinterpret_cast<T *>(smem);
    uint8_t *flg = smem + (size_t)S * VAL_BYTES;
    T *pack = reinterpret_cast<T *>(smem + (size_t)S * (VAL_BYTES + FLAG_BYTES));   // partition only
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * (VAL_BYTES + FLAG_BYTES) +
                                                  sel_pack_bytes<T, PARTITION>());
    uint64_t *empty = full + S;
    uint64_t *agg_done = empty + S;          // the rest: R slots, slot k % R
    uint64_t *prefix_ready = agg_done + R;
    long long *tile_of = reinterpret_cast<long long *>(prefix_ready + R);
    U *agg_of = reinterpret_cast<U *>(tile_of + R);
    U *excl_of = agg_of + R;
    __shared__ U s_warp[2][kSCW];
    __shared__ int s_abort;   // a compute warp's wait ran out: all of them leave

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    Header *hdr = reinterpret_cast<Header *>(a.ws);
    void *desc = a.ws + kHeaderBytes;
    const unsigned long long n = a.n;
    const T *in = reinterpret_cast<const T *>(a.in);
    const T thr = from_raw<T>(a.threshold_bits);

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
            mbar_init(&empty[s], kSCW + 1);
        }
        for (int slot = 0; slot < R; ++slot) {
            mbar_init(&agg_done[slot], 1);
            mbar_init(&prefix_ready[slot], 1);
            tile_of[slot] = num_tiles;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (!s_ok) return;   // same verdict in every CTA
    const uint32_t epoch = s_epoch;
    if (tid == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_HEADER);

    if (warp == kSCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int ends = 0;   // end markers sent: one per look-back warp
            for (long long k = 0;; ++k) {
                const int s = (int)(k % S);
                if (k >= S && !mbar_wait(&empty[s], (uint32_t)((k / S - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    break;
                }
                const long long t = ends ? num_tiles : (long long)atomicAdd(&hdr->tile_counter, 1ull);
                tile_of[k % R] = t;
                if (t < num_tiles) {
                    prefetch_descriptor<1>(desc, t);
                    PS_TRACE_POINT(t, PS_TRACE_CLAIM);
                    PS_TRACE_CTA(t);
                }
                if (a.use_bulk && t < num_tiles && (unsigned long long)(t + 1) * TILE <= n) {
                    mbar_arrive_expect_tx(&full[s], VAL_BYTES + FLAG_BYTES);
                    bulk_load(vals + (size_t)s * TILE, in + t * TILE, VAL_BYTES, &full[s]);
                    if (OP == 0) bulk_load(flg + (size_t)s * TILE, a.flags + t * TILE, FLAG_BYTES, &full[s]);
                } else {
                    mbar_arrive(&full[s]);   // end marker, or a tile read from global
                }
                if (t >= num_tiles && ++ends == LB) break;
            }
            if (epoch != kEpochMask) claims_done(hdr, a.ws_bytes, epoch);
        }
    } else if (warp == kSCW + 1) {
        // ---------------- aggregator: count and publish ----------------
        int ends = 0;   // end markers passed on: one per look-back warp
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!mbar_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const int slot = (int)(k % R);
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) {   // end marker: pass it on to the look-back warps
                if (lane == 0) mbar_arrive(&agg_done[slot]);
                if (++ends == LB) break;
                continue;
            }
            if (lane == 0) PS_TRACE_POINT(tile, PS_TRACE_DATA);
            const U cnt = count_tile<T, OP>(a, thr, vals + (size_t)s * TILE, flg + (size_t)s * TILE,
                                            (unsigned long long)tile * TILE, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const U agg = __reduce_add_sync(kFull, cnt);
            if (lane == 0) {
                Desc<U, 1>::store(desc, tile, tile == 0 ? kFlagP : kFlagA, agg, epoch);
                PS_TRACE_POINT(tile, PS_TRACE_AGGREGATE);
                agg_of[slot] = agg;
                mbar_arrive(&agg_done[slot]);
            }
        }
    } else if (warp >= kSCW + 2) {
        // ---------------- look-back warps: the tile's output offset ----------------
        // warp j takes iterations j, j + LB, ...
        for (long long k = warp - (kSCW + 2);; k += LB) {
            const int slot = (int)(k % R);
            if (!mbar_wait(&agg_done[slot], (uint32_t)((k / R) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            const U agg = agg_of[slot];
            if (lane == 0) PS_TRACE_POINT(tile, PS_TRACE_LOOKBACK_START);
            __syncwarp();
            U excl = 0;
            if (tile != 0) {
                excl = look_back<U, 1, kLookbackK>(desc, tile, epoch, a.max_polls, &hdr->status,
                                                   PS_TRACE_LOOKBACK(tile));
                if (lane == 0) Desc<U, 1>::store(desc, tile, kFlagP, excl + agg, epoch);
            }
            if (lane == 0) {
                if (a.num_selected && tile == num_tiles - 1) *a.num_selected = (unsigned long long)(excl + agg);
                excl_of[slot] = excl;
                PS_TRACE_POINT(tile, PS_TRACE_PREFIX);
                mbar_arrive(&prefix_ready[slot]);
            }
        }
    } else {
        // ---------------- compute warps: scan the flags, scatter ----------------
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!mbar_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                abort_meet(&s_abort, 1, CT);
                break;
            }
            const int slot = (int)(k % R);
            const long long tile = tile_of[slot];
            if (tile < 0 || tile >= num_tiles) break;
            const auto wait_prefix = [&]() -> U {
                if (!mbar_wait(&prefix_ready[slot], (uint32_t)((k / R) & 1)))
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                return excl_of[slot];
            };
            if (!select_tile_pass<T, OP, PARTITION>(a, thr, tile, vals + (size_t)s * TILE, flg + (size_t)s * TILE,
                                                    pack, &empty[s], s_warp[k & 1], &s_abort, wait_prefix))
                break;
        }
        if (warp == 0 && lane == 0) PS_TRACE_CTA_POINT(PS_TRACE_CTA_DONE);
    }

    // the last producer readied the workspace; before an epoch wrap the
    // last CTA to finish does
    if (epoch == kEpochMask) finish_call(hdr, a.ws, a.ws_bytes, epoch);
}

// ---- paired tiles -------------------------------------------------------------
// The same operation with one look-back per two tiles: the two CTAs of a
// cluster take tiles 2u and 2u+1 as one unit u (one claim and one
// descriptor per unit), each copying and scanning its own tile at the same
// time.  CTA 0 (the leader) claims the unit and passes its id to CTA 1;
// CTA 1 passes its tile's count back; the leader publishes the unit's
// count, looks back over the units, publishes P, and hands CTA 1 the
// offset of its tile (the unit's offset plus the leader's count) -- all
// through distributed shared memory, with bounded waits.  Half the
// descriptors and look-backs per byte; CTA 1 runs none.  An odd number of
// tiles leaves CTA 1 an empty tile in the last unit.  In place is safe as
// before: a tile learns its offset after every earlier unit and the leader's
// own tile have published their counts, which each does after its data sits
// in shared memory.
#ifndef PS_SEL_PAIR
#define PS_SEL_PAIR 0
#endif
template <typename T, int OP, bool PARTITION> constexpr size_t sel_pair_smem_bytes() {
    // unit id and its mailbox, partner's and own count, and three mbarriers
    // per hand-off slot
    return sel_smem_bytes<T, OP, PARTITION>() + ((size_t)sel_ring<OP, PARTITION>() * 48 + 127) / 128 * 128;
}

template <typename T, int OP, bool PARTITION>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(sel_threads<PARTITION>(), kSCtasPerSm)
select_pair_kernel(SelectArgs a, long long num_tiles) {
    using U = uint32_t;                     // counts
    constexpr int VEC = Traits<T>::VEC;
    constexpr int ITEMS = SelItems<T>::value;
    constexpr long long TILE = sel_tile<T>();
    constexpr int S = sel_stages<OP, PARTITION>();
    constexpr int R = sel_ring<OP, PARTITION>();
    constexpr uint32_t VAL_BYTES = (uint32_t)(TILE * sizeof(T));
    constexpr uint32_t FLAG_BYTES = OP == 0 ? (uint32_t)TILE : 0u;
    constexpr int CT = kSCW * 32;
    constexpr int LB = sel_lookback_warps<PARTITION>();
    static_assert(ITEMS % VEC == 0, "ITEMS must be a multiple of the vector width");
    static_assert(LB <= S, "at most one look-back warp per stage");
    static_assert(R % 2 == 0, "8-byte alignment of the hand-off slots");
    const long long num_units = (num_tiles + 1) / 2;

    extern __shared__ __align__(128) unsigned char smem[];
    T *vals = reinterpret_cast<T *>(smem);
    uint8_t *flg = smem + (size_t)S * VAL_BYTES;
    T *pack = reinterpret_cast<T *>(smem + (size_t)S * (VAL_BYTES + FLAG_BYTES));   // partition only
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * (VAL_BYTES + FLAG_BYTES) +
                                                  sel_pack_bytes<T, PARTITION>());
    uint64_t *empty = full + S;
    uint64_t *agg_done = empty + S;          // the rest: R slots, slot k % R
    uint64_t *prefix_ready = agg_done + R;
    long long *tile_of = reinterpret_cast<long long *>(prefix_ready + R);
    U *agg_of = reinterpret_cast<U *>(tile_of + R);   // the leader: the unit's count
    U *excl_of = agg_of + R;
    long long *unit_of = reinterpret_cast<long long *>(excl_of + R);   // written by this CTA's producer
    long long *unit_box = unit_of + R;                // CTA 1: the leader writes the unit id here
    U *part_of = reinterpret_cast<U *>(unit_box + R); // the leader: CTA 1's count
    U *own_of = part_of + R;                          // the leader: its own tile's count
    uint64_t *unit_rdy = reinterpret_cast<uint64_t *>(own_of + R);   // CTA 1: unit id arrived
    uint64_t *unit_free = unit_rdy + R;                              // leader: CTA 1 has read it
    uint64_t *part_rdy = unit_free + R;                              // leader: CTA 1's count arrived
    __shared__ U s_warp[2][kSCW];
    __shared__ int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    Header *hdr = reinterpret_cast<Header *>(a.ws);
    void *desc = a.ws + kHeaderBytes;
    const unsigned long long n = a.n;
    const T *in = reinterpret_cast<const T *>(a.in);
    const T thr = from_raw<T>(a.threshold_bits);

    __shared__ uint32_t s_epoch;
    __shared__ int s_ok;
    if (tid == 0) {
        uint32_t e;
        s_ok = begin_call(hdr, &e) ? 1 : 0;
        s_epoch = e;
        s_abort = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kSCW + 1);
        }
        for (int slot = 0; slot < R; ++slot) {
            mbar_init(&agg_done[slot], 1);
            mbar_init(&prefix_ready[slot], 1);
            mbar_init(&unit_rdy[slot], 1);
            mbar_init(&unit_free[slot], 1);
            mbar_init(&part_rdy[slot], 1);
            tile_of[slot] = num_tiles;
            unit_of[slot] = num_units;
            unit_box[slot] = num_units;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers are ready before either arrives on the other's
    if (!s_ok) return;    // the same verdict in both CTAs of the cluster (one header)
    const uint32_t epoch = s_epoch;

    if (warp == kSCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            int ends = 0;   // end markers: one per look-back warp in the leader, one in CTA 1
            for (long long k = 0;; ++k) {
                const int s = (int)(k % S);
                const int slot = (int)(k % R);
                if (k >= S && !mbar_wait(&empty[s], (uint32_t)((k / S - 1) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    break;
                }
                long long u;
                if (rank == 0) {
                    u = ends ? num_units : (long long)atomicAdd(&hdr->tile_counter, 1ull);
                    if (ends == 0) {
                        // CTA 1 follows the same units: pass the id on, once it
                        // has read the one this slot held R iterations ago
                        if (k >= R && !mbar_wait_cluster(&unit_free[slot], (uint32_t)((k / R - 1) & 1))) {
                            report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                            break;
                        }
                        st_cluster_u64(cluster_addr(&unit_box[slot], 1), (unsigned long long)u);
                        mbar_arrive_cluster(cluster_addr(&unit_rdy[slot], 1));
                    }
                    if (u < num_units) prefetch_descriptor<1>(desc, u);
                } else {
                    // the leader may refill the mailbox as soon as this
                    // iteration has read it; the CTA's other warps read the
                    // local copy, which only this producer writes
                    if (!mbar_wait_cluster(&unit_rdy[slot], (uint32_t)((k / R) & 1))) {
                        report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                        break;
                    }
                    u = unit_box[slot];
                    mbar_arrive_cluster(cluster_addr(&unit_free[slot], 0));
                }
                unit_of[slot] = u;
                const long long t = u < num_units ? 2 * u + (long long)rank : num_tiles;
                tile_of[slot] = t;
                if (a.use_bulk && t < num_tiles && (unsigned long long)(t + 1) * TILE <= n) {
                    mbar_arrive_expect_tx(&full[s], VAL_BYTES + FLAG_BYTES);
                    bulk_load(vals + (size_t)s * TILE, in + t * TILE, VAL_BYTES, &full[s]);
                    if (OP == 0) bulk_load(flg + (size_t)s * TILE, a.flags + t * TILE, FLAG_BYTES, &full[s]);
                } else {
                    mbar_arrive(&full[s]);   // end marker, an empty tile, or one read from global
                }
                if (u >= num_units && (rank == 1 || ++ends == LB)) break;
            }
            if (epoch != kEpochMask) claims_done(hdr, a.ws_bytes, epoch);
        }
    } else if (warp == kSCW + 1) {
        // ---------------- aggregator: count; the leader publishes the unit's ----------------
        int ends = 0;
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!mbar_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                break;
            }
            const int slot = (int)(k % R);
            const long long u = unit_of[slot];
            const long long tile = tile_of[slot];
            if (u >= num_units) {   // end marker: pass it on to the look-back warps
                if (lane == 0) mbar_arrive(&agg_done[slot]);
                if (rank == 1 || ++ends == LB) break;
                continue;
            }
            // CTA 1's empty tile (past the array) counts nothing
            const U cnt = count_tile<T, OP>(a, thr, vals + (size_t)s * TILE, flg + (size_t)s * TILE,
                                            (unsigned long long)tile * TILE, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            const U agg = __reduce_add_sync(kFull, cnt);
            if (lane == 0) {
                if (rank == 1) {
                    st_cluster_u32(cluster_addr(&part_of[slot], 0), agg);
                    mbar_arrive_cluster(cluster_addr(&part_rdy[slot], 0));
                } else {
                    U pc = 0;
                    if (mbar_wait_cluster(&part_rdy[slot], (uint32_t)((k / R) & 1)))
                        pc = part_of[slot];
                    else
                        report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    Desc<U, 1>::store(desc, u, u == 0 ? kFlagP : kFlagA, agg + pc, epoch);
                    own_of[slot] = agg;
                    agg_of[slot] = agg + pc;
                    mbar_arrive(&agg_done[slot]);
                }
            }
        }
    } else if (warp >= kSCW + 2) {
        // ---------------- look-back warps (the leader): the unit's offset ----------------
        if (rank == 0) {
            for (long long k = warp - (kSCW + 2);; k += LB) {
                const int slot = (int)(k % R);
                if (!mbar_wait(&agg_done[slot], (uint32_t)((k / R) & 1))) {
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                    break;
                }
                const long long u = unit_of[slot];
                if (u >= num_units) break;
                const U agg = agg_of[slot];
                __syncwarp();
                U excl = 0;
                if (u != 0) {
                    excl = look_back<U, 1, kLookbackK>(desc, u, epoch, a.max_polls, &hdr->status);
                    if (lane == 0) Desc<U, 1>::store(desc, u, kFlagP, excl + agg, epoch);
                }
                if (lane == 0) {
                    if (a.num_selected && u == num_units - 1) *a.num_selected = (unsigned long long)(excl + agg);
                    excl_of[slot] = excl;
                    mbar_arrive(&prefix_ready[slot]);
                    // CTA 1's tile follows the leader's in the unit
                    st_cluster_u32(cluster_addr(&excl_of[slot], 1), excl + own_of[slot]);
                    mbar_arrive_cluster(cluster_addr(&prefix_ready[slot], 1));
                }
            }
        }
    } else {
        // ---------------- compute warps: scan the flags, scatter ----------------
        for (long long k = 0;; ++k) {
            const int s = (int)(k % S);
            if (!mbar_wait(&full[s], (uint32_t)((k / S) & 1))) {
                report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                abort_meet(&s_abort, 1, CT);
                break;
            }
            const int slot = (int)(k % R);
            if (unit_of[slot] >= num_units) break;
            // CTA 1's offset comes from the leader: acquire at cluster scope
            const auto wait_prefix = [&]() -> U {
                if (!mbar_wait_cluster(&prefix_ready[slot], (uint32_t)((k / R) & 1)))
                    report_error(&hdr->status, epoch, PS_ERR_LOOKBACK_TIMEOUT);
                return excl_of[slot];
            };
            if (!select_tile_pass<T, OP, PARTITION>(a, thr, tile_of[slot], vals + (size_t)s * TILE,
                                                    flg + (size_t)s * TILE, pack, &empty[s], s_warp[k & 1],
                                                    &s_abort, wait_prefix))
                break;
        }
    }

    // no CTA leaves while its partner may still write to its shared memory
    cluster_sync_all();
    if (epoch == kEpochMask) finish_call(hdr, a.ws, a.ws_bytes, epoch);
}

template <typename T, int OP, bool PARTITION>
static cudaError_t launch_select_variant(const SelectArgs &a, cudaStream_t s) {
    constexpr bool kPair = PS_SEL_PAIR != 0;
    constexpr size_t smem = kPair ? sel_pair_smem_bytes<T, OP, PARTITION>() : sel_smem_bytes<T, OP, PARTITION>();
    const long long tiles = (long long)((a.n + sel_tile<T>() - 1) / sel_tile<T>());
    static volatile int configured[64] = {};
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        if constexpr (kPair)
            e = cudaFuncSetAttribute(select_pair_kernel<T, OP, PARTITION>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        else
            e = cudaFuncSetAttribute(select_kernel<T, OP, PARTITION>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    long long grid = (long long)sms * kSCtasPerSm;
    if constexpr (kPair) {
        // clusters of two CTAs, one per unit of two tiles
        const long long units = (tiles + 1) / 2;
        if (grid > 2 * units) grid = 2 * units;
        grid &= ~1ll;
        select_pair_kernel<T, OP, PARTITION><<<(unsigned int)grid, sel_threads<PARTITION>(), smem, s>>>(a, tiles);
    } else {
        if (grid > tiles) grid = tiles;
        select_kernel<T, OP, PARTITION><<<(unsigned int)grid, sel_threads<PARTITION>(), smem, s>>>(a, tiles);
    }
    return cudaGetLastError();
}

template <typename T, bool PARTITION>
static cudaError_t launch_select_part(const SelectArgs &a, int op, cudaStream_t s) {
    switch (op) {
    case 0: return launch_select_variant<T, 0, PARTITION>(a, s);
    case 1: return launch_select_variant<T, 1, PARTITION>(a, s);
    case 2: return launch_select_variant<T, 2, PARTITION>(a, s);
    default: return launch_select_variant<T, 3, PARTITION>(a, s);
    }
}

template <typename T>
cudaError_t launch_select(const SelectArgs &a, int op, bool partition, cudaStream_t s) {
    return partition ? launch_select_part<T, true>(a, op, s) : launch_select_part<T, false>(a, op, s);
}

template cudaError_t launch_select<int32_t>(const SelectArgs &, int, bool, cudaStream_t);
template cudaError_t launch_select<int64_t>(const SelectArgs &, int, bool, cudaStream_t);
template cudaError_t launch_select<float>(const SelectArgs &, int, bool, cudaStream_t);

TRACE_COPY_FUNCTIONS(trace_copy_select, trace_copy_select_ctas)

}  // namespace ps
