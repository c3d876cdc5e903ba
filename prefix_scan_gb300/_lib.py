"""ctypes binding of ``libprefixscan.so`` (argument marshalling only).

The names and signatures mirror ``include/prefix_scan.h`` and
``include/prefix_scan_testing.h`` one to one.  Nothing here computes: every
step of a scan runs in the CUDA library.  Loading fails loudly when the
library has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import threading

from .build import LIBRARY

PS_OK = 0
PS_ERR_INVALID_ARG = 1
PS_ERR_WORKSPACE_TOO_SMALL = 2
PS_ERR_OVERLAP = 3
PS_ERR_CUDA = 4
PS_ERR_LOOKBACK_TIMEOUT = 5
PS_ERR_WORKSPACE_NOT_INITIALIZED = 6

PS_INT32, PS_INT64, PS_FLOAT32 = 0, 1, 2
PS_ALGO_DECOUPLED_LOOKBACK, PS_ALGO_REDUCE_THEN_SCAN, PS_ALGO_CHAINED = 0, 1, 2
PS_FLAG_X, PS_FLAG_A, PS_FLAG_P = 0, 1, 2

_vp, _sz, _int, _u32, _i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32, ctypes.c_int64

# name -> (restype, argtypes); one entry per declaration in include/*.h
SIGNATURES = {
    "ps_scan_workspace_size": (_sz, [_int, _sz]),
    "ps_tile_elements": (_sz, [_int]),
    "ps_scan": (_int, [_int, _int, _int, _vp, _vp, _sz, _vp, _sz, _vp]),
    "ps_get_device_status": (_int, [_vp, _vp, ctypes.POINTER(_int)]),
    "ps_status_string": (ctypes.c_char_p, [_int]),
    "ps_last_cuda_error": (_int, []),
    "ps_testing_descriptor_bytes": (_sz, [_int]),
    "ps_testing_encode_descriptor": (_int, [_int, _int, _u32, _vp, _vp]),
    "ps_testing_lookback": (_int, [_int, _vp, _i64, _u32, _u32, _vp, _vp, _vp]),
    "ps_testing_workspace_epoch": (_int, [_vp, _vp, ctypes.POINTER(_u32)]),
    "ps_testing_set_workspace_epoch": (_int, [_vp, _u32, _vp]),
    "ps_workspace_init": (_int, [_vp, _sz, _vp]),
}
SIGNATURES["ps_scan_inclusive_i32_noalloc"] = (_int, [_vp, _vp, _sz, _vp])
SIGNATURES["ps_testing_noalloc_scratch"] = (_int, [ctypes.POINTER(_vp), _vp])
SIGNATURES["ps_trace_capacity"] = (_sz, [])
SIGNATURES["ps_trace_read"] = (_int, [_int, _vp, _vp, _vp, _sz])
SIGNATURES["ps_trace_read_ctas"] = (_int, [_int, _vp, _sz])
SIGNATURES["ps_scan_seeded"] = (_int, [_int, _int, _vp, _vp, _sz, _vp, _vp, _vp, _sz, _vp])
SIGNATURES["ps_scan_host_staging_size"] = (_sz, [_int, _sz])
SIGNATURES["ps_scan_host"] = (_int, [_int, _int, _vp, _vp, _sz, _vp, _sz, _vp, _sz, _vp])
SIGNATURES["ps_scan_op"] = (_int, [_int, _int, _int, _vp, _vp, _sz, _vp, _sz, _vp])
PS_OP_SUM, PS_OP_MAX, PS_OP_MIN = 0, 1, 2
SIGNATURES["ps_select"] = (_int, [_int, _int, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp])
SIGNATURES["ps_partition"] = (_int, [_int, _int, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp])
PS_SELECT_FLAGGED, PS_SELECT_NONZERO, PS_SELECT_GREATER, PS_SELECT_LESS = 0, 1, 2, 3
SIGNATURES["ps_scan_pair_i32_f32"] = (_int, [_int, _vp, _vp, _sz, _vp, _sz, _vp])
SIGNATURES["ps_scan_affine_f32"] = (_int, [_int, _vp, _vp, _sz, _vp, _sz, _vp])
SIGNATURES["ps_reduce_by_key_workspace_size"] = (_sz, [_int, _sz])
SIGNATURES["ps_reduce_by_key"] = (_int, [_int, _int, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp])
SIGNATURES["ps_run_length_encode"] = (_int, [_int, _vp, _vp, _vp, _vp, _sz, _vp, _sz, _vp])
PS_NOALLOC_MAX_ELEMENTS = 1 << 29

for _kind in ("inclusive", "exclusive"):
    for _t in ("i32", "i64", "f32"):
        SIGNATURES[f"ps_scan_{_kind}_{_t}"] = (_int, [_vp, _vp, _sz, _vp, _sz, _vp])

_lock = threading.Lock()
_lib = None


class PrefixScanError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = status_string(status)
        extra = f" (cudaError {cuda_error})" if status == PS_ERR_CUDA else ""
        super().__init__(f"{fn} failed: {name}{extra}")


def load() -> ctypes.CDLL:
    """Load the CUDA library, raising if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not LIBRARY.exists():
                raise RuntimeError(
                    f"{LIBRARY} is not built; run prefix_scan_gb300.build.build() "
                    "(or __graft_entry__.build()) first")
            lib = ctypes.CDLL(str(LIBRARY))
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    try:
        return load().ps_status_string(status).decode()
    except Exception:  # the library itself may be what failed to load
        return f"status {status}"


def check(fn: str, status: int) -> None:
    if status != PS_OK:
        raise PrefixScanError(fn, status, load().ps_last_cuda_error() if status == PS_ERR_CUDA else 0)
