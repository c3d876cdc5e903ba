"""CPU oracle for the prefix sum -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never touches it and
it never touches the CUDA library: the two share no code.

The arithmetic lives in ``scan_oracle.c`` (a plain sequential running sum,
written from the definition y[i] = x[0] + ... + x[i] on the cumsum page
"CUDA-Operators-6-Cumsum", section 1, and the inclusive/exclusive conversion
section of the RTX 4090 scan tutorial; and a plain sequential stream
compaction, the definition behind section 4.4 of the decoupled look-back
paper summary).  This module only compiles that file with gcc and marshals
numpy arrays into it.

Every function here is pinned by ``tests/test_oracle_pins.py``; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "scan_oracle.c"
LIBRARY = _HERE / "_scan_oracle.so"

_lock = threading.Lock()
_lib = None

_INT_TYPES = {
    np.dtype(np.int32): ("i32", ctypes.c_int32),
    np.dtype(np.int64): ("i64", ctypes.c_int64),
}


def build(force: bool = False, source: Path | None = None, target: Path | None = None) -> Path:
    """Compile the oracle with gcc into a shared object (no-op when fresh).

    ``source``/``target`` let a test compile a modified copy elsewhere.
    """
    src = Path(source) if source is not None else SOURCE
    out = Path(target) if target is not None else LIBRARY
    if not force and out.exists() and out.stat().st_mtime >= src.stat().st_mtime:
        return out
    tmp = out.with_name(out.name + f".{os.getpid()}.tmp")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared",
           "-o", str(tmp), str(src), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    for name in ("oracle_inclusive_i32", "oracle_exclusive_i32",
                 "oracle_inclusive_i64", "oracle_exclusive_i64",
                 "oracle_inclusive_f32", "oracle_exclusive_f32"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, sz, vp]
        fn.restype = None
    lib.oracle_abs_prefix_f32.argtypes = [vp, sz, ctypes.c_int, vp]
    lib.oracle_abs_prefix_f32.restype = None
    for name in ("oracle_select_b32", "oracle_select_b64", "oracle_partition_b32",
                 "oracle_partition_b64"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, sz, vp]
        fn.restype = sz
    lib.oracle_flags_i32.argtypes = [vp, sz, ctypes.c_int, ctypes.c_int32, vp]
    lib.oracle_flags_i64.argtypes = [vp, sz, ctypes.c_int, ctypes.c_int64, vp]
    lib.oracle_flags_f32.argtypes = [vp, sz, ctypes.c_int, ctypes.c_float, vp]
    for fn in (lib.oracle_flags_i32, lib.oracle_flags_i64, lib.oracle_flags_f32):
        fn.restype = None
    for name in ("oracle_scan_op_i32", "oracle_scan_op_i64", "oracle_scan_op_f32"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, sz, ctypes.c_int, ctypes.c_int, vp]
        fn.restype = None
    for name in ("oracle_rbk_b32_i32", "oracle_rbk_b64_i32"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, sz, vp, vp]
        fn.restype = sz
    for name in ("oracle_rbk_b32_f32", "oracle_rbk_b64_f32"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, vp, sz, vp, vp, vp]
        fn.restype = sz
    lib.oracle_scan_pair_i32_f32.argtypes = [vp, vp, sz, ctypes.c_int, vp, vp, vp]
    lib.oracle_scan_pair_i32_f32.restype = None
    lib.oracle_scan_affine_f32.argtypes = [vp, vp, sz, ctypes.c_int, vp, vp, vp, vp]
    lib.oracle_scan_affine_f32.restype = None
    return lib


def load(path: Path | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the compiled oracle."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(str(path)))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(str(build())))
        return _lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _scan(x: np.ndarray, exclusive: bool, lib: ctypes.CDLL | None) -> np.ndarray:
    lib = lib if lib is not None else load()
    x = np.ascontiguousarray(x)
    kind = "exclusive" if exclusive else "inclusive"
    if x.dtype == np.float32:
        y = np.empty(x.shape[0], dtype=np.float64)
        getattr(lib, f"oracle_{kind}_f32")(_ptr(x), x.shape[0], _ptr(y))
        return y
    if x.dtype not in _INT_TYPES:
        raise TypeError(f"oracle: unsupported dtype {x.dtype}")
    tag, _ = _INT_TYPES[x.dtype]
    y = np.empty_like(x)
    getattr(lib, f"oracle_{kind}_{tag}")(_ptr(x), x.shape[0], _ptr(y))
    return y


def inclusive(x: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """y[i] = x[0] + ... + x[i]; int32/int64 wrap modulo 2^w, fp32 -> float64."""
    return _scan(x, False, lib)


def exclusive(x: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """y[0] = 0, y[i] = x[0] + ... + x[i-1]; same types as :func:`inclusive`."""
    return _scan(x, True, lib)


def abs_prefix(x: np.ndarray, exclusive_: bool, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Prefix sums of |x| in float64 (the scale of the fp32 error bound)."""
    lib = lib if lib is not None else load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    a = np.empty(x.shape[0], dtype=np.float64)
    lib.oracle_abs_prefix_f32(_ptr(x), x.shape[0], int(bool(exclusive_)), _ptr(a))
    return a


# ---- stream compaction -------------------------------------------------------

PREDICATES = {"nonzero": 0, "greater": 1, "less": 2}


def flags(x: np.ndarray, op: str, threshold=0, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """uint8 flags of a value predicate: nonzero, greater (x > t), less (x < t)."""
    lib = lib if lib is not None else load()
    x = np.ascontiguousarray(x)
    f = np.empty(x.shape[0], dtype=np.uint8)
    fn = {np.dtype(np.int32): lib.oracle_flags_i32, np.dtype(np.int64): lib.oracle_flags_i64,
          np.dtype(np.float32): lib.oracle_flags_f32}[x.dtype]
    fn(_ptr(x), x.shape[0], PREDICATES[op], threshold, _ptr(f))
    return f


def _compact(x: np.ndarray, f: np.ndarray, partition: bool, lib) -> tuple[np.ndarray, int]:
    lib = lib if lib is not None else load()
    x = np.ascontiguousarray(x)
    f = np.ascontiguousarray(f, dtype=np.uint8)
    if f.shape != x.shape:
        raise ValueError("oracle: flags and values differ in length")
    out = np.zeros_like(x)
    bits = x.dtype.itemsize * 8
    name = f"oracle_{'partition' if partition else 'select'}_b{bits}"
    k = int(getattr(lib, name)(_ptr(x), _ptr(f), x.shape[0], _ptr(out)))
    return out, k


def select(x: np.ndarray, f: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """The elements of x whose flag is nonzero, in order."""
    out, k = _compact(x, f, False, lib)
    return out[:k]


def partition(x: np.ndarray, f: np.ndarray, lib: ctypes.CDLL | None = None) -> tuple[np.ndarray, int]:
    """Flagged elements first in order, the others from the back in reverse; (out, count)."""
    return _compact(x, f, True, lib)


# ---- running maximum / minimum -------------------------------------------------

OPS = {"max": 1, "min": 2}


def scan_op(x: np.ndarray, op: str, exclusive_: bool = False,
            lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Running max / min (inclusive, or exclusive with the identity first)."""
    lib = lib if lib is not None else load()
    x = np.ascontiguousarray(x)
    y = np.empty_like(x)
    fn = {np.dtype(np.int32): lib.oracle_scan_op_i32, np.dtype(np.int64): lib.oracle_scan_op_i64,
          np.dtype(np.float32): lib.oracle_scan_op_f32}[x.dtype]
    fn(_ptr(x), x.shape[0], OPS[op], int(bool(exclusive_)), _ptr(y))
    return y


# ---- reduce-by-key / run-length encoding ---------------------------------------


def reduce_by_key(keys: np.ndarray, values: np.ndarray | None = None,
                  lib: ctypes.CDLL | None = None):
    """Runs of bitwise-equal consecutive keys: (unique keys, per-run values).

    values int32 -> int32 run sums (mod 2^32); values fp32 -> (float64 run
    sums, float64 run sums of |value|); values None -> int32 run lengths.
    """
    lib = lib if lib is not None else load()
    keys = np.ascontiguousarray(keys)
    n = keys.shape[0]
    bits = keys.dtype.itemsize * 8
    kraw = keys.view(np.uint32 if bits == 32 else np.uint64)
    okeys = np.empty(n, dtype=kraw.dtype)
    if values is None or values.dtype == np.int32:
        vals = None if values is None else np.ascontiguousarray(values)
        if vals is not None and vals.shape[0] != n:
            raise ValueError("oracle: keys and values differ in length")
        ov = np.empty(n, dtype=np.int32)
        m = getattr(lib, f"oracle_rbk_b{bits}_i32")(_ptr(kraw), _ptr(vals) if vals is not None else None,
                                                     n, _ptr(okeys), _ptr(ov))
        return okeys[:m].view(keys.dtype), ov[:m]
    vals = np.ascontiguousarray(values, dtype=np.float32)
    ov = np.empty(n, dtype=np.float64)
    oa = np.empty(n, dtype=np.float64)
    m = getattr(lib, f"oracle_rbk_b{bits}_f32")(_ptr(kraw), _ptr(vals), n, _ptr(okeys), _ptr(ov), _ptr(oa))
    return okeys[:m].view(keys.dtype), ov[:m], oa[:m]


# ---- pair scans ------------------------------------------------------------------


def scan_pair_i32_f32(xi: np.ndarray, xf: np.ndarray, exclusive: bool = False,
                      lib: ctypes.CDLL | None = None):
    """{int32, fp32} pairs summed field by field: (int32 sums mod 2^32,
    float64 sums, float64 running sums of |f|)."""
    lib = lib if lib is not None else load()
    xi = np.ascontiguousarray(xi, dtype=np.int32)
    xf = np.ascontiguousarray(xf, dtype=np.float32)
    n = xi.shape[0]
    if xf.shape[0] != n:
        raise ValueError("oracle: pair fields differ in length")
    yi = np.empty(n, dtype=np.int32)
    yf = np.empty(n, dtype=np.float64)
    ya = np.empty(n, dtype=np.float64)
    lib.oracle_scan_pair_i32_f32(_ptr(xi), _ptr(xf), n, int(exclusive), _ptr(yi), _ptr(yf), _ptr(ya))
    return yi, yf, ya


def scan_affine_f32(a: np.ndarray, b: np.ndarray, exclusive: bool = False,
                    lib: ctypes.CDLL | None = None):
    """Composition of the maps x -> a_k x + b_k in input order: (A, B, |A|,
    |B|-scale), all float64."""
    lib = lib if lib is not None else load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    n = a.shape[0]
    if b.shape[0] != n:
        raise ValueError("oracle: map fields differ in length")
    out = [np.empty(n, dtype=np.float64) for _ in range(4)]
    lib.oracle_scan_affine_f32(_ptr(a), _ptr(b), n, int(exclusive), *[_ptr(o) for o in out])
    return tuple(out)
