// scan_api.cu -- the library's C ABI: argument checks, workspace sizing,
// dispatch to the launchers, status reporting.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>

#include "prefix_scan.h"
#include "prefix_scan_testing.h"
#include "prefix_scan_trace.h"
#include "scan_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

ps_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return PS_ERR_CUDA;
}

bool valid_dtype(int dt) { return dt == PS_INT32 || dt == PS_INT64 || dt == PS_FLOAT32; }

// Do byte ranges [a, a+an) and [b, b+bn) intersect?
bool ranges_overlap(const void *a, size_t an, const void *b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

ps_status check_args(ps_dtype dt, const void *in, const void *out, size_t n, const void *ws,
                     size_t ws_bytes) {
    if (!valid_dtype(dt)) return PS_ERR_INVALID_ARG;
    if (in == nullptr || out == nullptr || ws == nullptr) return PS_ERR_INVALID_ARG;
    const size_t es = ps::elem_bytes(dt);
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % es != 0)
        return PS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return PS_ERR_INVALID_ARG;
    if (n > (SIZE_MAX / 2) / es) return PS_ERR_INVALID_ARG;
    if (ps::num_tiles(dt, n) > (size_t)INT_MAX) return PS_ERR_INVALID_ARG;
    if (ws_bytes < ps::workspace_bytes(dt, n)) return PS_ERR_WORKSPACE_TOO_SMALL;
    const size_t bytes = n * es;
    if (in != out && ranges_overlap(in, bytes, out, bytes)) return PS_ERR_OVERLAP;
    const size_t wsb = ps::workspace_bytes(dt, n);
    if (ranges_overlap(ws, wsb, in, bytes) || ranges_overlap(ws, wsb, out, bytes)) return PS_ERR_OVERLAP;
    return PS_OK;
}

template <typename T>
ps_status run(ps_algo algo, bool exclusive, const void *in, void *out, size_t n, void *ws,
              size_t ws_bytes, cudaStream_t s, const void *carry_in = nullptr,
              void *carry_out = nullptr, int op = ps::kOpSum) {
    cudaError_t e;
    unsigned char *w = static_cast<unsigned char *>(ws);
    switch (algo) {
    case PS_ALGO_DECOUPLED_LOOKBACK:
    case PS_ALGO_CHAINED: {
        ps::PassArgs a{in, out, (unsigned long long)n, w, carry_in, carry_out,
                       (unsigned long long)(ws_bytes & ~(size_t)7), ps::kDefaultMaxPolls};
        e = ps::launch_single_pass<T>(a, exclusive,
                                      algo == PS_ALGO_CHAINED ? ps::Lookback::Chained
                                                              : ps::Lookback::Decoupled, s, op);
        break;
    }
    case PS_ALGO_REDUCE_THEN_SCAN:
        e = ps::launch_reduce_then_scan<T>(in, out, (unsigned long long)n, w, exclusive, s);
        break;
    default:
        return PS_ERR_INVALID_ARG;
    }
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

ps_status dispatch(ps_algo algo, ps_dtype dt, int exclusive, const void *in, void *out, size_t n,
                   void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!valid_dtype(dt)) return PS_ERR_INVALID_ARG;
    if (algo != PS_ALGO_DECOUPLED_LOOKBACK && algo != PS_ALGO_REDUCE_THEN_SCAN && algo != PS_ALGO_CHAINED)
        return PS_ERR_INVALID_ARG;
    if (n == 0) return PS_OK;
    const ps_status st = check_args(dt, in, out, n, ws, ws_bytes);
    if (st != PS_OK) return st;
    switch (dt) {
    case PS_INT32: return run<int32_t>(algo, exclusive != 0, in, out, n, ws, ws_bytes, s);
    case PS_INT64: return run<int64_t>(algo, exclusive != 0, in, out, n, ws, ws_bytes, s);
    case PS_FLOAT32: return run<float>(algo, exclusive != 0, in, out, n, ws, ws_bytes, s);
    }
    return PS_ERR_INVALID_ARG;
}

}  // namespace

void ps::note_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

namespace {

ps_status compact(bool partition, ps_dtype dt, int op, const void *in, const uint8_t *flags,
                  const void *threshold, void *out, uint64_t *num_selected, size_t n, void *ws,
                  size_t ws_bytes, cudaStream_t s) {
    if (!valid_dtype(dt) || op < PS_SELECT_FLAGGED || op > PS_SELECT_LESS) return PS_ERR_INVALID_ARG;
    const size_t es = ps::elem_bytes(dt);
    if (reinterpret_cast<uintptr_t>(num_selected) % 8 != 0) return PS_ERR_INVALID_ARG;
    if (n == 0) {
        if (num_selected == nullptr) return PS_OK;
        const cudaError_t e = cudaMemsetAsync(num_selected, 0, sizeof(uint64_t), s);
        return e == cudaSuccess ? PS_OK : cuda_fail(e);
    }
    if (n > 0xffffffffull) return PS_ERR_INVALID_ARG;   // 32-bit counts
    if (op == PS_SELECT_FLAGGED && flags == nullptr) return PS_ERR_INVALID_ARG;
    if ((op == PS_SELECT_GREATER || op == PS_SELECT_LESS) && threshold == nullptr) return PS_ERR_INVALID_ARG;
    const ps_status st = check_args(dt, in, out, n, ws, ws_bytes);
    if (st != PS_OK) return st;
    const size_t bytes = n * es;
    const bool bulk = ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(flags)) & 15u) == 0;
    if (in == out && (partition || !bulk)) return PS_ERR_OVERLAP;   // see ps_select / ps_partition
    if (op == PS_SELECT_FLAGGED && (ranges_overlap(flags, n, out, bytes) ||
                                    ranges_overlap(flags, n, ws, ps::workspace_bytes(dt, n))))
        return PS_ERR_OVERLAP;
    if (num_selected && (ranges_overlap(num_selected, 8, out, bytes) || ranges_overlap(num_selected, 8, in, bytes) ||
                         ranges_overlap(num_selected, 8, ws, ps::workspace_bytes(dt, n))))
        return PS_ERR_OVERLAP;
    unsigned long long tb = 0;
    if (threshold) std::memcpy(&tb, threshold, es);
    ps::SelectArgs a{in, op == PS_SELECT_FLAGGED ? flags : nullptr, out, (unsigned long long)n,
                     static_cast<unsigned char *>(ws), (unsigned long long)(ws_bytes & ~(size_t)7),
                     reinterpret_cast<unsigned long long *>(num_selected), tb, ps::kDefaultMaxPolls,
                     bulk ? 1 : 0};
    cudaError_t e;
    switch (dt) {
    case PS_INT32: e = ps::launch_select<int32_t>(a, op, partition, s); break;
    case PS_INT64: e = ps::launch_select<int64_t>(a, op, partition, s); break;
    default: e = ps::launch_select<float>(a, op, partition, s); break;
    }
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

ps_status reduce_by_key(ps_dtype kdt, ps_dtype vdt, bool rle, const void *keys, const void *vals,
                        void *ukeys, void *aggs, uint64_t *num_runs, size_t n, void *ws,
                        size_t ws_bytes, cudaStream_t s) {
    if (!valid_dtype(kdt) || (vdt != PS_INT32 && vdt != PS_FLOAT32)) return PS_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(num_runs) % 8 != 0) return PS_ERR_INVALID_ARG;
    if (n == 0) {
        if (num_runs == nullptr) return PS_OK;
        const cudaError_t e = cudaMemsetAsync(num_runs, 0, sizeof(uint64_t), s);
        return e == cudaSuccess ? PS_OK : cuda_fail(e);
    }
    if (n > 0xffffffffull) return PS_ERR_INVALID_ARG;   // 32-bit run counts
    if (keys == nullptr || ukeys == nullptr || aggs == nullptr || ws == nullptr || (!rle && vals == nullptr))
        return PS_ERR_INVALID_ARG;
    const size_t kes = ps::elem_bytes(kdt);
    if ((reinterpret_cast<uintptr_t>(keys) | reinterpret_cast<uintptr_t>(ukeys)) % kes != 0 ||
        (reinterpret_cast<uintptr_t>(vals) | reinterpret_cast<uintptr_t>(aggs)) % 4 != 0 ||
        reinterpret_cast<uintptr_t>(ws) % 16 != 0)
        return PS_ERR_INVALID_ARG;
    if (ps::rbk_num_tiles(kdt, n) > (size_t)INT_MAX) return PS_ERR_INVALID_ARG;
    const size_t wsb = ps::rbk_workspace_bytes(kdt, n);
    if (ws_bytes < wsb) return PS_ERR_WORKSPACE_TOO_SMALL;
    const size_t kb = n * kes, vb = n * 4;
    struct Range { const void *p; size_t b; };
    const Range ins[] = {{keys, kb}, {rle ? nullptr : vals, vb}};
    const Range outs[] = {{ukeys, kb}, {aggs, vb}, {ws, wsb}, {num_runs, num_runs ? 8u : 0u}};
    for (const Range &o : outs) {
        if (o.p == nullptr) continue;
        for (const Range &i : ins)
            if (i.p && ranges_overlap(o.p, o.b, i.p, i.b)) return PS_ERR_OVERLAP;
        for (const Range &o2 : outs)
            if (&o2 != &o && o2.p && ranges_overlap(o.p, o.b, o2.p, o2.b)) return PS_ERR_OVERLAP;
    }
    const bool bulk = ((reinterpret_cast<uintptr_t>(keys) | reinterpret_cast<uintptr_t>(rle ? nullptr : vals)) & 15u) == 0;
    ps::RbkArgs a{keys, rle ? nullptr : vals, ukeys, aggs, (unsigned long long)n,
                  static_cast<unsigned char *>(ws), (unsigned long long)(ws_bytes & ~(size_t)7),
                  reinterpret_cast<unsigned long long *>(num_runs), ps::kDefaultMaxPolls, bulk ? 1 : 0};
    const cudaError_t e = rle ? ps::launch_run_length_encode(a, kdt, s) : ps::launch_reduce_by_key(a, kdt, vdt, s);
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

}  // namespace

ps_status ps::scan_seeded(ps_dtype dt, int exclusive, const void *in, void *out, size_t n,
                          const void *carry_in, void *carry_out, void *ws, size_t ws_bytes,
                          cudaStream_t s) {
    if (!valid_dtype(dt)) return PS_ERR_INVALID_ARG;
    const size_t es = ps::elem_bytes(dt);
    if ((reinterpret_cast<uintptr_t>(carry_in) | reinterpret_cast<uintptr_t>(carry_out)) % es != 0)
        return PS_ERR_INVALID_ARG;
    if (n == 0) {
        // the running total of nothing added to carry_in is carry_in
        if (carry_out == nullptr || carry_out == carry_in) return PS_OK;
        cudaError_t e = carry_in ? cudaMemcpyAsync(carry_out, carry_in, es, cudaMemcpyDeviceToDevice, s)
                                 : cudaMemsetAsync(carry_out, 0, es, s);
        return e == cudaSuccess ? PS_OK : cuda_fail(e);
    }
    const ps_status st = check_args(dt, in, out, n, ws, ws_bytes);
    if (st != PS_OK) return st;
    const size_t bytes = n * es, wsb = ps::workspace_bytes(dt, n);
    for (const void *c : {static_cast<const void *>(carry_in), static_cast<const void *>(carry_out)})
        if (c && (ranges_overlap(c, es, in, bytes) || ranges_overlap(c, es, out, bytes) ||
                  ranges_overlap(c, es, ws, wsb)))
            return PS_ERR_OVERLAP;
    switch (dt) {
    case PS_INT32: return run<int32_t>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes, s, carry_in, carry_out);
    case PS_INT64: return run<int64_t>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes, s, carry_in, carry_out);
    case PS_FLOAT32: return run<float>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes, s, carry_in, carry_out);
    }
    return PS_ERR_INVALID_ARG;
}

extern "C" {

size_t ps_scan_workspace_size(ps_dtype dtype, size_t n) {
    if (!valid_dtype(dtype)) return 0;
    return ps::workspace_bytes(dtype, n);
}

size_t ps_tile_elements(ps_dtype dtype) {
    if (!valid_dtype(dtype)) return 0;
    return ps::tile_elems(dtype);
}

ps_status ps_scan(ps_algo algo, ps_dtype dtype, int exclusive, const void *in, void *out, size_t n,
                  void *ws, size_t ws_bytes, ps_stream_t stream) {
    return dispatch(algo, dtype, exclusive, in, out, n, ws, ws_bytes, (cudaStream_t)stream);
}

#define PS_DEFINE_ENTRY(NAME, CTYPE, DT, EXCL)                                                   \
    ps_status NAME(const CTYPE *in, CTYPE *out, size_t n, void *ws, size_t ws_bytes,             \
                   ps_stream_t stream) {                                                         \
        return dispatch(PS_ALGO_DECOUPLED_LOOKBACK, DT, EXCL, in, out, n, ws, ws_bytes,          \
                        (cudaStream_t)stream);                                                   \
    }
PS_DEFINE_ENTRY(ps_scan_inclusive_i32, int32_t, PS_INT32, 0)
PS_DEFINE_ENTRY(ps_scan_exclusive_i32, int32_t, PS_INT32, 1)
PS_DEFINE_ENTRY(ps_scan_inclusive_i64, int64_t, PS_INT64, 0)
PS_DEFINE_ENTRY(ps_scan_exclusive_i64, int64_t, PS_INT64, 1)
PS_DEFINE_ENTRY(ps_scan_inclusive_f32, float, PS_FLOAT32, 0)
PS_DEFINE_ENTRY(ps_scan_exclusive_f32, float, PS_FLOAT32, 1)
#undef PS_DEFINE_ENTRY

ps_status ps_scan_seeded(ps_dtype dtype, int exclusive, const void *in, void *out, size_t n,
                         const void *carry_in, void *carry_out, void *ws, size_t ws_bytes,
                         ps_stream_t stream) {
    return ps::scan_seeded(dtype, exclusive, in, out, n, carry_in, carry_out, ws, ws_bytes,
                           (cudaStream_t)stream);
}

ps_status ps_scan_op(ps_op op, ps_dtype dtype, int exclusive, const void *in, void *out, size_t n,
                     void *ws, size_t ws_bytes, ps_stream_t stream) {
    if (!valid_dtype(dtype) || (op != PS_OP_SUM && op != PS_OP_MAX && op != PS_OP_MIN))
        return PS_ERR_INVALID_ARG;
    if (n == 0) return PS_OK;
    const ps_status st = check_args(dtype, in, out, n, ws, ws_bytes);
    if (st != PS_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    switch (dtype) {
    case PS_INT32: return run<int32_t>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes, s, nullptr, nullptr, op);
    case PS_INT64: return run<int64_t>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes, s, nullptr, nullptr, op);
    default: return run<float>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes, s, nullptr, nullptr, op);
    }
}

ps_status ps_scan_pair_i32_f32(int exclusive, const ps_pair_i32_f32 *in, ps_pair_i32_f32 *out, size_t n,
                               void *ws, size_t ws_bytes, ps_stream_t stream) {
    if (n == 0) return PS_OK;
    const ps_status st = check_args(PS_INT64, in, out, n, ws, ws_bytes);   // 8-byte elements
    if (st != PS_OK) return st;
    return run<int64_t>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes,
                        (cudaStream_t)stream, nullptr, nullptr, ps::kOpPairI32F32);
}

ps_status ps_scan_affine_f32(int exclusive, const ps_affine_f32 *in, ps_affine_f32 *out, size_t n, void *ws,
                             size_t ws_bytes, ps_stream_t stream) {
    if (n == 0) return PS_OK;
    const ps_status st = check_args(PS_INT64, in, out, n, ws, ws_bytes);
    if (st != PS_OK) return st;
    return run<int64_t>(PS_ALGO_DECOUPLED_LOOKBACK, exclusive != 0, in, out, n, ws, ws_bytes,
                        (cudaStream_t)stream, nullptr, nullptr, ps::kOpAffineF32);
}

ps_status ps_select(ps_dtype dtype, ps_select_op op, const void *in, const uint8_t *flags,
                    const void *threshold, void *out, uint64_t *num_selected, size_t n, void *ws,
                    size_t ws_bytes, ps_stream_t stream) {
    return compact(false, dtype, (int)op, in, flags, threshold, out, num_selected, n, ws, ws_bytes,
                   (cudaStream_t)stream);
}

ps_status ps_partition(ps_dtype dtype, ps_select_op op, const void *in, const uint8_t *flags,
                       const void *threshold, void *out, uint64_t *num_selected, size_t n, void *ws,
                       size_t ws_bytes, ps_stream_t stream) {
    return compact(true, dtype, (int)op, in, flags, threshold, out, num_selected, n, ws, ws_bytes,
                   (cudaStream_t)stream);
}

size_t ps_reduce_by_key_workspace_size(ps_dtype key_dtype, size_t n) {
    if (!valid_dtype(key_dtype)) return 0;
    return ps::rbk_workspace_bytes(key_dtype, n);
}

ps_status ps_reduce_by_key(ps_dtype key_dtype, ps_dtype value_dtype, const void *keys,
                           const void *values, void *unique_keys, void *aggregates,
                           uint64_t *num_runs, size_t n, void *ws, size_t ws_bytes,
                           ps_stream_t stream) {
    return reduce_by_key(key_dtype, value_dtype, false, keys, values, unique_keys, aggregates, num_runs,
                         n, ws, ws_bytes, (cudaStream_t)stream);
}

ps_status ps_run_length_encode(ps_dtype key_dtype, const void *keys, void *unique_keys,
                               int32_t *counts, uint64_t *num_runs, size_t n, void *ws,
                               size_t ws_bytes, ps_stream_t stream) {
    return reduce_by_key(key_dtype, PS_INT32, true, keys, nullptr, unique_keys, counts, num_runs, n, ws,
                         ws_bytes, (cudaStream_t)stream);
}

ps_status ps_workspace_init(void *ws, size_t ws_bytes, ps_stream_t stream) {
    if (ws_bytes == 0) return PS_OK;
    if (ws == nullptr || reinterpret_cast<uintptr_t>(ws) % 16 != 0) return PS_ERR_INVALID_ARG;
    const cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream);
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

ps_status ps_get_device_status(const void *ws, ps_stream_t stream, ps_status *out) {
    if (ws == nullptr || out == nullptr) return PS_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e);
    ps::Header h;
    e = cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!((h.magic == ps::kWorkspaceMagic && h.epoch <= ps::kEpochMask) || (h.magic == 0 && h.epoch == 0))) {
        *out = PS_ERR_WORKSPACE_NOT_INITIALIZED;
        return PS_OK;
    }
    // the last call that completed ran as epoch - 1; older errors are history
    const uint32_t last = (h.epoch - 1u) & ps::kEpochMask;
    const bool current = h.magic == ps::kWorkspaceMagic && (uint32_t)(h.status >> 8) == last;
    *out = current ? (ps_status)(h.status & 0xffu) : PS_OK;
    return PS_OK;
}

const char *ps_status_string(ps_status status) {
    switch (status) {
    case PS_OK: return "PS_OK";
    case PS_ERR_INVALID_ARG: return "PS_ERR_INVALID_ARG";
    case PS_ERR_WORKSPACE_TOO_SMALL: return "PS_ERR_WORKSPACE_TOO_SMALL";
    case PS_ERR_OVERLAP: return "PS_ERR_OVERLAP";
    case PS_ERR_CUDA: return "PS_ERR_CUDA";
    case PS_ERR_LOOKBACK_TIMEOUT: return "PS_ERR_LOOKBACK_TIMEOUT";
    case PS_ERR_WORKSPACE_NOT_INITIALIZED: return "PS_ERR_WORKSPACE_NOT_INITIALIZED";
    }
    return "PS_ERR_UNKNOWN";
}

int ps_last_cuda_error(void) { return g_last_cuda_error; }

// ---- test hooks -------------------------------------------------------------

size_t ps_testing_descriptor_bytes(ps_dtype dtype) {
    if (!valid_dtype(dtype)) return 0;
    return ps::desc_bytes(dtype);
}

ps_status ps_testing_encode_descriptor(ps_dtype dtype, int flag, uint32_t epoch, const void *value,
                                       void *out) {
    if (!valid_dtype(dtype) || value == nullptr || out == nullptr || epoch > ps::kEpochMask)
        return PS_ERR_INVALID_ARG;
    if (flag != PS_FLAG_X && flag != PS_FLAG_A && flag != PS_FLAG_P) return PS_ERR_INVALID_ARG;
    const uint64_t t = ((uint64_t)epoch << 34) | ((uint64_t)flag << 32);
    if (dtype == PS_INT64) {
        uint64_t v;
        std::memcpy(&v, value, 8);
        const uint64_t w[2] = {t | (v & 0xffffffffull), t | (v >> 32)};
        std::memcpy(out, w, 16);
    } else {
        uint32_t v;
        std::memcpy(&v, value, 4);
        const uint64_t w = t | v;
        std::memcpy(out, &w, 8);
    }
    return PS_OK;
}

ps_status ps_testing_lookback(ps_dtype dtype, const void *desc, int64_t tile, uint32_t epoch,
                              uint32_t max_polls, void *result, uint64_t *status,
                              ps_stream_t stream) {
    if (!valid_dtype(dtype) || desc == nullptr || result == nullptr || status == nullptr || tile < 1 ||
        epoch > ps::kEpochMask)
        return PS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned long long *st = reinterpret_cast<unsigned long long *>(status);
    cudaError_t e;
    switch (dtype) {
    case PS_INT32: e = ps::launch_lookback_probe<int32_t>(desc, tile, epoch, max_polls, result, st, s); break;
    case PS_INT64: e = ps::launch_lookback_probe<int64_t>(desc, tile, epoch, max_polls, result, st, s); break;
    default: e = ps::launch_lookback_probe<float>(desc, tile, epoch, max_polls, result, st, s); break;
    }
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

ps_status ps_testing_workspace_epoch(const void *ws, ps_stream_t stream, uint32_t *epoch) {
    if (ws == nullptr || epoch == nullptr) return PS_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpy(epoch, static_cast<const unsigned char *>(ws) + offsetof(ps::Header, epoch),
                       sizeof(uint32_t), cudaMemcpyDeviceToHost);
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

ps_status ps_testing_set_workspace_epoch(void *ws, uint32_t epoch, ps_stream_t stream) {
    if (ws == nullptr || epoch > ps::kEpochMask) return PS_ERR_INVALID_ARG;
    const uint32_t magic = ps::kWorkspaceMagic;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpy(static_cast<unsigned char *>(ws) + offsetof(ps::Header, epoch), &epoch,
                       sizeof(uint32_t), cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
        e = cudaMemcpy(static_cast<unsigned char *>(ws) + offsetof(ps::Header, magic), &magic,
                       sizeof(uint32_t), cudaMemcpyHostToDevice);
    return e == cudaSuccess ? PS_OK : cuda_fail(e);
}

}  // extern "C"

// ---- pipeline trace (include/prefix_scan_trace.h) ----------------------------
extern "C" size_t ps_trace_capacity(void) {
#ifdef PS_TRACE
    return (size_t)PS_TRACE_TILES;
#else
    return 0;
#endif
}

extern "C" ps_status ps_trace_read(int kernel, uint64_t *timestamps, uint32_t *lookback, int32_t *cta,
                                   size_t tiles) {
#ifdef PS_TRACE
    if (timestamps == nullptr || lookback == nullptr || cta == nullptr || tiles > (size_t)PS_TRACE_TILES)
        return PS_ERR_INVALID_ARG;
    if (tiles == 0) return PS_OK;
    cudaError_t e;
    switch (kernel) {
    case PS_TRACE_KERNEL_SCAN: e = ps::trace_copy_scan(timestamps, lookback, cta, tiles); break;
    case PS_TRACE_KERNEL_SELECT: e = ps::trace_copy_select(timestamps, lookback, cta, tiles); break;
    case PS_TRACE_KERNEL_RBK: e = ps::trace_copy_rbk(timestamps, lookback, cta, tiles); break;
    case PS_TRACE_KERNEL_RLE: e = ps::trace_copy_rle(timestamps, lookback, cta, tiles); break;
    default: return PS_ERR_INVALID_ARG;
    }
    if (e != cudaSuccess) {
        ps::note_cuda_error(e);
        return PS_ERR_CUDA;
    }
    return PS_OK;
#else
    (void)kernel, (void)timestamps, (void)lookback, (void)cta, (void)tiles;
    return PS_ERR_INVALID_ARG;   // this build records no trace
#endif
}

extern "C" ps_status ps_trace_read_ctas(int kernel, uint64_t *timestamps, size_t ctas) {
#ifdef PS_TRACE
    if (timestamps == nullptr || ctas > (size_t)PS_TRACE_CTAS) return PS_ERR_INVALID_ARG;
    if (ctas == 0) return PS_OK;
    cudaError_t e;
    switch (kernel) {
    case PS_TRACE_KERNEL_SCAN: e = ps::trace_copy_scan_ctas(timestamps, ctas); break;
    case PS_TRACE_KERNEL_SELECT: e = ps::trace_copy_select_ctas(timestamps, ctas); break;
    case PS_TRACE_KERNEL_RBK: e = ps::trace_copy_rbk_ctas(timestamps, ctas); break;
    case PS_TRACE_KERNEL_RLE: e = ps::trace_copy_rle_ctas(timestamps, ctas); break;
    default: return PS_ERR_INVALID_ARG;
    }
    if (e != cudaSuccess) {
        ps::note_cuda_error(e);
        return PS_ERR_CUDA;
    }
    return PS_OK;
#else
    (void)kernel, (void)timestamps, (void)ctas;
    return PS_ERR_INVALID_ARG;   // this build records no trace
#endif
}
