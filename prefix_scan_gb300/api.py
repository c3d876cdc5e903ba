"""PyTorch-facing wrappers of the C ABI.

PyTorch only supplies device memory and streams here: tensors are passed to
the library as raw device pointers with the current (or given) CUDA stream,
and every step of the scan runs in ``libprefixscan.so``.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (PS_ALGO_CHAINED, PS_ALGO_DECOUPLED_LOOKBACK, PS_ALGO_REDUCE_THEN_SCAN,
                   PS_FLOAT32, PS_INT32, PS_INT64)

DTYPE_CODES = {torch.int32: PS_INT32, torch.int64: PS_INT64, torch.float32: PS_FLOAT32}
_SUFFIX = {PS_INT32: "i32", PS_INT64: "i64", PS_FLOAT32: "f32"}
ALGOS = {"decoupled": PS_ALGO_DECOUPLED_LOOKBACK,
         "reduce_then_scan": PS_ALGO_REDUCE_THEN_SCAN,
         # fixed association: bitwise-reproducible fp32 results
         "deterministic": PS_ALGO_REDUCE_THEN_SCAN,
         "chained": PS_ALGO_CHAINED}


def dtype_code(dtype: torch.dtype) -> int:
    try:
        return DTYPE_CODES[dtype]
    except KeyError:
        raise TypeError(f"prefix scan supports int32, int64 and float32, not {dtype}") from None


def workspace_size(dtype: torch.dtype, n: int) -> int:
    """Bytes of device workspace a scan of ``n`` elements needs."""
    return int(_lib.load().ps_scan_workspace_size(dtype_code(dtype), n))


def tile_elements(dtype: torch.dtype) -> int:
    return int(_lib.load().ps_tile_elements(dtype_code(dtype)))


def alloc_workspace(dtype: torch.dtype, n: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 device tensor large enough for a scan of ``n``
    elements, ready for any number of calls (it must not be reused for
    anything else in between)."""
    return torch.zeros(max(workspace_size(dtype, n), 16), dtype=torch.uint8, device=device or "cuda")


def _stream_handle(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


OPS = {"sum": 0, "max": 1, "min": 2}


def scan(x: torch.Tensor, *, exclusive: bool = False, out: torch.Tensor | None = None,
         inplace: bool = False, workspace: torch.Tensor | None = None, stream=None,
         algo: str = "decoupled", op: str = "sum") -> torch.Tensor:
    """Inclusive/exclusive sum scan of a contiguous 1-D CUDA tensor.

    ``inplace=True`` writes the result over ``x``.  ``workspace`` (uint8,
    on the same device) is allocated when not given.  The call is
    asynchronous on ``stream`` (default: the current stream).
    """
    if not x.is_cuda:
        raise ValueError("prefix scan: input must be a CUDA tensor (there is no CPU path)")
    if x.dim() != 1 or not x.is_contiguous():
        raise ValueError("prefix scan: input must be a contiguous 1-D tensor")
    code = dtype_code(x.dtype)
    n = x.numel()
    if inplace:
        if out is not None and out.data_ptr() != x.data_ptr():
            raise ValueError("prefix scan: inplace=True and a distinct `out` are exclusive")
        out = x
    elif out is None:
        out = torch.empty_like(x)
    elif out.dtype != x.dtype or out.numel() != n or not out.is_contiguous() or out.device != x.device:
        raise ValueError("prefix scan: `out` must match the input's dtype, length and device")
    if n == 0:
        return out
    lib = _lib.load()
    need = int(lib.ps_scan_workspace_size(code, n))
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    elif workspace.numel() * workspace.element_size() < need or workspace.device != x.device:
        raise ValueError(f"prefix scan: workspace needs {need} bytes on {x.device}")
    ws_bytes = workspace.numel() * workspace.element_size()
    s = _stream_handle(stream, x.device)
    if op != "sum":
        if algo != "decoupled":
            raise ValueError("prefix scan: max/min scans run the decoupled look-back only")
        name = "ps_scan_op"
        st = lib.ps_scan_op(OPS[op], code, int(exclusive), x.data_ptr(), out.data_ptr(), n,
                            workspace.data_ptr(), ws_bytes, s)
    elif algo == "decoupled":
        kind = "exclusive" if exclusive else "inclusive"
        name = f"ps_scan_{kind}_{_SUFFIX[code]}"
        st = getattr(lib, name)(x.data_ptr(), out.data_ptr(), n, workspace.data_ptr(), ws_bytes, s)
    else:
        name = "ps_scan"
        st = lib.ps_scan(ALGOS[algo], code, int(exclusive), x.data_ptr(), out.data_ptr(), n,
                         workspace.data_ptr(), ws_bytes, s)
    _lib.check(name, st)
    return out


def scan_inclusive(x: torch.Tensor, out: torch.Tensor | None = None, **kw) -> torch.Tensor:
    """y[i] = x[0] + ... + x[i] (device-wide, single pass)."""
    return scan(x, exclusive=False, out=out, **kw)


def scan_exclusive(x: torch.Tensor, out: torch.Tensor | None = None, **kw) -> torch.Tensor:
    """y[0] = 0, y[i] = x[0] + ... + x[i-1] (device-wide, single pass)."""
    return scan(x, exclusive=True, out=out, **kw)


def scan_seeded(x: torch.Tensor, carry_in: torch.Tensor | None = None,
                carry_out: torch.Tensor | None = None, *, exclusive: bool = False,
                out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Scan with a device carry: y = carry_in + scan(x); carry_out = carry_in + sum(x).

    ``carry_in``/``carry_out`` are one-element CUDA tensors of x's dtype (or
    None); they may be the same tensor.
    """
    if not x.is_cuda or x.dim() != 1 or not x.is_contiguous():
        raise ValueError("prefix scan: input must be a contiguous 1-D CUDA tensor")
    code = dtype_code(x.dtype)
    n = x.numel()
    out = torch.empty_like(x) if out is None else out
    for c in (carry_in, carry_out):
        if c is not None and (c.dtype != x.dtype or c.numel() != 1 or c.device != x.device):
            raise ValueError("prefix scan: carries are one-element tensors of the input's dtype")
    lib = _lib.load()
    need = int(lib.ps_scan_workspace_size(code, n))
    if workspace is None:
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=x.device)
    st = lib.ps_scan_seeded(code, int(exclusive), x.data_ptr() if n else None,
                            out.data_ptr() if n else None, n,
                            carry_in.data_ptr() if carry_in is not None else None,
                            carry_out.data_ptr() if carry_out is not None else None,
                            workspace.data_ptr(), workspace.numel(), _stream_handle(stream, x.device))
    _lib.check("ps_scan_seeded", st)
    return out


SELECT_OPS = {"flagged": 0, "nonzero": 1, "greater": 2, "less": 3}


def _compact(partition: bool, x: torch.Tensor, flags, op, threshold, out, inplace, workspace, stream):
    if not x.is_cuda or x.dim() != 1 or not x.is_contiguous():
        raise ValueError("select: input must be a contiguous 1-D CUDA tensor")
    code = dtype_code(x.dtype)
    n = x.numel()
    op = op or ("flagged" if flags is not None else "nonzero")
    if op == "flagged":
        if flags is None or flags.dtype != torch.uint8 or flags.numel() != n or not flags.is_cuda:
            raise ValueError("select: `flags` must be a uint8 CUDA tensor of the input's length")
    if inplace:
        out = x
    elif out is None:
        out = torch.empty_like(x)
    count = torch.zeros(1, dtype=torch.int64, device=x.device)
    lib = _lib.load()
    need = int(lib.ps_scan_workspace_size(code, n))
    if workspace is None:
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=x.device)
    thr = None
    if threshold is not None:
        import numpy as np
        thr = np.array([threshold], dtype={torch.int32: np.int32, torch.int64: np.int64,
                                           torch.float32: np.float32}[x.dtype])
    fn = lib.ps_partition if partition else lib.ps_select
    st = fn(code, SELECT_OPS[op], x.data_ptr() if n else None,
            flags.data_ptr() if (flags is not None and n) else None,
            thr.ctypes.data if thr is not None else None, out.data_ptr() if n else None,
            count.data_ptr(), n, workspace.data_ptr(), workspace.numel(), _stream_handle(stream, x.device))
    _lib.check("ps_partition" if partition else "ps_select", st)
    return out, count


def select(x: torch.Tensor, flags: torch.Tensor | None = None, *, op: str | None = None,
           threshold=None, out: torch.Tensor | None = None, inplace: bool = False,
           workspace: torch.Tensor | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Single-pass stream compaction: (out, count) with the kept elements in
    out[:count] in input order.  ``op``: "flagged" (flags != 0), "nonzero",
    "greater"/"less" (than ``threshold``).  ``count`` is a one-element int64
    CUDA tensor (no host synchronisation here)."""
    return _compact(False, x, flags, op, threshold, out, inplace, workspace, stream)


def partition(x: torch.Tensor, flags: torch.Tensor | None = None, *, op: str | None = None,
              threshold=None, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Kept elements to out[:count] in order, the others to the back in
    reverse order (out[n-1-j] = j-th rejected)."""
    return _compact(True, x, flags, op, threshold, out, False, workspace, stream)


def _pair_scan(fname: str, x: torch.Tensor, exclusive: bool, out, inplace: bool, workspace, stream):
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError(f"{fname}: input must be a contiguous CUDA tensor")
    if x.dim() == 2 and x.shape[1] == 2 and x.element_size() == 4:
        n = x.shape[0]
    elif x.dim() == 1 and x.element_size() == 8:
        n = x.shape[0]
    else:
        raise ValueError(f"{fname}: expected (n, 2) 32-bit elements or (n,) 8-byte elements")
    if inplace:
        out = x
    elif out is None:
        out = torch.empty_like(x)
    if out.data_ptr() != x.data_ptr() and (out.numel() * out.element_size() != n * 8 or not out.is_contiguous()):
        raise ValueError(f"{fname}: `out` must hold n 8-byte elements")
    lib = _lib.load()
    if workspace is None:
        workspace = alloc_workspace(torch.int64, n, x.device)
    if n:
        st = getattr(lib, fname)(int(exclusive), x.data_ptr(), out.data_ptr(), n, workspace.data_ptr(),
                                 workspace.numel(), _stream_handle(stream, x.device))
        _lib.check(fname, st)
    return out


def scan_pairs(x: torch.Tensor, *, exclusive: bool = False, out: torch.Tensor | None = None,
               inplace: bool = False, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Scan of {int32, fp32} pairs summed field by field.  ``x``: an (n,)
    int64 tensor holding the pairs' bits (int32 field in the low half), or
    an (n, 2) int32 tensor whose second column holds the fp32 bits."""
    return _pair_scan("ps_scan_pair_i32_f32", x, exclusive, out, inplace, workspace, stream)


def scan_affine(x: torch.Tensor, *, exclusive: bool = False, out: torch.Tensor | None = None,
                inplace: bool = False, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Composition scan of the fp32 affine maps x -> a x + b given as an
    (n, 2) float32 tensor of rows (a, b); row k of the result is the
    composition of maps 0..k (map 0 applied first)."""
    return _pair_scan("ps_scan_affine_f32", x, exclusive, out, inplace, workspace, stream)


def reduce_by_key_workspace_size(key_dtype: torch.dtype, n: int) -> int:
    return int(_lib.load().ps_reduce_by_key_workspace_size(dtype_code(key_dtype), n))


def _runs(keys: torch.Tensor, values, unique_keys, aggregates, workspace, stream, num_runs=None):
    if not keys.is_cuda or keys.dim() != 1 or not keys.is_contiguous():
        raise ValueError("reduce_by_key: keys must be a contiguous 1-D CUDA tensor")
    n = keys.numel()
    kcode = dtype_code(keys.dtype)
    if values is not None:
        if (not values.is_cuda or values.dim() != 1 or not values.is_contiguous() or values.numel() != n
                or values.dtype not in (torch.int32, torch.float32)):
            raise ValueError("reduce_by_key: values must be a contiguous int32/fp32 CUDA tensor "
                             "of the keys' length")
    adt = values.dtype if values is not None else torch.int32
    if unique_keys is None:
        unique_keys = torch.empty_like(keys)
    if aggregates is None:
        aggregates = torch.empty(n, dtype=adt, device=keys.device)
    if unique_keys.dtype != keys.dtype or unique_keys.numel() < n or aggregates.dtype != adt or aggregates.numel() < n:
        raise ValueError("reduce_by_key: outputs need n entries of the key / aggregate dtype")
    if num_runs is None:
        num_runs = torch.zeros(1, dtype=torch.int64, device=keys.device)
    elif not num_runs.is_cuda or num_runs.dtype != torch.int64 or num_runs.numel() < 1:
        raise ValueError("reduce_by_key: num_runs must be an int64 CUDA tensor of at least one entry")
    lib = _lib.load()
    if workspace is None:
        need = int(lib.ps_reduce_by_key_workspace_size(kcode, n))
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=keys.device)
    sh = _stream_handle(stream, keys.device)
    ptr = (lambda t: t.data_ptr() if n else None)
    if values is None:
        st = lib.ps_run_length_encode(kcode, ptr(keys), ptr(unique_keys), ptr(aggregates), num_runs.data_ptr(),
                                      n, workspace.data_ptr(), workspace.numel(), sh)
        _lib.check("ps_run_length_encode", st)
    else:
        st = lib.ps_reduce_by_key(kcode, dtype_code(values.dtype), ptr(keys), ptr(values), ptr(unique_keys),
                                  ptr(aggregates), num_runs.data_ptr(), n, workspace.data_ptr(),
                                  workspace.numel(), sh)
        _lib.check("ps_reduce_by_key", st)
    return unique_keys, aggregates, num_runs


def reduce_by_key(keys: torch.Tensor, values: torch.Tensor, *, unique_keys: torch.Tensor | None = None,
                  aggregates: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None, num_runs: torch.Tensor | None = None
                  ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Single-pass reduce-by-key: for each run of consecutive bitwise-equal
    keys, its key and the sum of its values.  Returns (unique_keys,
    aggregates, num_runs): full-length outputs whose first ``num_runs``
    entries are defined; ``num_runs`` is a one-element int64 CUDA tensor
    (no host synchronisation here), allocated when not given."""
    if values is None:
        raise ValueError("reduce_by_key: values are required (run_length_encode counts runs)")
    return _runs(keys, values, unique_keys, aggregates, workspace, stream, num_runs)


def run_length_encode(keys: torch.Tensor, *, unique_keys: torch.Tensor | None = None,
                      counts: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None, num_runs: torch.Tensor | None = None
                      ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Single-pass run-length encoding: (unique_keys, counts, num_runs) as
    for :func:`reduce_by_key`, with int32 run lengths."""
    return _runs(keys, None, unique_keys, counts, workspace, stream, num_runs)


def host_staging_size(dtype: torch.dtype, n: int) -> int:
    return int(_lib.load().ps_scan_host_staging_size(dtype_code(dtype), n))


class HostScanBuffers:
    """Device staging buffer + workspace for :func:`scan_host`, reusable across calls."""

    def __init__(self, dtype: torch.dtype, n: int, device=None):
        dev = torch.device(device or "cuda")
        self.dtype, self.n = dtype, n
        self.staging = torch.empty(max(host_staging_size(dtype, n), 256), dtype=torch.uint8, device=dev)
        self.workspace = torch.zeros(max(workspace_size(dtype, n), 16), dtype=torch.uint8, device=dev)


def scan_host(x: torch.Tensor, *, exclusive: bool = False, out: torch.Tensor | None = None,
              buffers: HostScanBuffers | None = None, stream=None, synchronize: bool = True,
              device=None) -> torch.Tensor:
    """Scan of a contiguous 1-D HOST tensor, streamed through the GPU.

    ``out`` (host) may be ``x`` for an in-place scan.  Pinned (page-locked)
    tensors let the two copy directions overlap.  With ``synchronize`` the
    call waits for the stream, so ``out`` is ready on return.
    """
    if x.is_cuda or x.dim() != 1 or not x.is_contiguous():
        raise ValueError("scan_host: input must be a contiguous 1-D host tensor")
    code = dtype_code(x.dtype)
    n = x.numel()
    out = torch.empty_like(x) if out is None else out
    if out.is_cuda or out.dtype != x.dtype or out.numel() != n or not out.is_contiguous():
        raise ValueError("scan_host: `out` must be a host tensor matching the input")
    if n == 0:
        return out
    dev = torch.device(device or "cuda")
    if buffers is None or buffers.n < n or buffers.dtype != x.dtype:
        buffers = HostScanBuffers(x.dtype, n, dev)
    s = stream if stream is not None else torch.cuda.current_stream(buffers.staging.device)
    st = _lib.load().ps_scan_host(code, int(exclusive), x.data_ptr(), out.data_ptr(), n,
                                  buffers.staging.data_ptr(), buffers.staging.numel(),
                                  buffers.workspace.data_ptr(), buffers.workspace.numel(),
                                  ctypes.c_void_p(s.cuda_stream))
    _lib.check("ps_scan_host", st)
    if synchronize:
        s.synchronize()
    return out


def device_status(workspace: torch.Tensor, stream=None) -> int:
    """Waits for the stream, returns the status the last scan left in ``workspace``."""
    lib = _lib.load()
    st = ctypes.c_int(0)
    _lib.check("ps_get_device_status",
               lib.ps_get_device_status(workspace.data_ptr(), _stream_handle(stream, workspace.device),
                                        ctypes.byref(st)))
    return st.value
