"""Seeded synthetic inputs for the prefix sum (host side).

This module is the only code that the CUDA path and the CPU oracle have in
common: it produces input arrays and nothing else.  It holds none of the
scan's arithmetic.

Generator: a counter-based hash.  Element ``i`` of a stream with seed ``s``
is ``splitmix64(key(s) + (i + 1) * 0x9E3779B97F4A7C15)`` where ``splitmix64``
is the output function of the SplitMix64 generator (Steele, Lea & Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014) and
``key(s) = splitmix64(s * 0x9E3779B97F4A7C15 + 0x632BE59BD9B4E019)``.  Being
counter-based, any slice can be produced independently, so large arrays are
filled in parallel chunks (plain C in ``csrc/inputs_gen.c``, one chunk per
thread; :func:`hash_block` is the same definition in numpy, kept for spot
checks of the C fill).

Value maps from the 64-bit hash ``h``:
  uniform integers in [lo, hi]   lo + (((h >> 32) * (hi - lo + 1)) >> 32)
                                 (multiply-shift range reduction, Lemire,
                                 "Fast random integer generation in an
                                 interval", ACM TOMACS 2019; span <= 2^32)
  Bernoulli(1/2) in {0, 1}       h >> 63
  fp32 uniform in [-1, 1)        (h >> 40) * 2^-23 - 1   (exact in fp32)
  full-range int32               low 32 bits, reinterpreted as int32
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_SEED_SALT = 0x632BE59BD9B4E019
_M64 = (1 << 64) - 1
_CHUNK = 1 << 22

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "csrc" / "inputs_gen.c"
_SO = _HERE / "_inputs_gen.so"
_lock = threading.Lock()
_lib = None


def build_generator(force: bool = False) -> Path:
    """Compile the C fill with gcc (no-op when fresh)."""
    if not force and _SO.exists() and _SO.stat().st_mtime >= _SRC.stat().st_mtime:
        return _SO
    tmp = _SO.with_name(_SO.name + f".{os.getpid()}.tmp")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(tmp), str(_SRC)],
                   check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build_generator()))
            u64, sz, vp, i64 = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int64
            lib.gen_hash_u64.argtypes = [u64, u64, sz, vp]
            lib.gen_uniform_i32.argtypes = [u64, u64, sz, i64, u64, vp]
            lib.gen_uniform_i64.argtypes = [u64, u64, sz, i64, u64, vp]
            lib.gen_bernoulli.argtypes = [u64, u64, sz, ctypes.c_int, vp]
            lib.gen_uniform_f32.argtypes = [u64, u64, sz, vp]
            lib.gen_full_i32.argtypes = [u64, u64, sz, vp]
            for f in (lib.gen_hash_u64, lib.gen_uniform_i32, lib.gen_uniform_i64,
                      lib.gen_bernoulli, lib.gen_uniform_f32, lib.gen_full_i32):
                f.restype = None
            _lib = lib
        return _lib


def _mix_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def seed_key(seed: int) -> int:
    return _mix_int(seed * GOLDEN + _SEED_SALT)


def hash_block(seed: int, start: int, count: int, key: int | None = None) -> np.ndarray:
    """Hashes of elements ``start .. start+count-1`` (numpy, for spot checks)."""
    z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    z *= np.uint64(GOLDEN)
    z += np.uint64(seed_key(seed) if key is None else key)
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def _fill(out: np.ndarray, call) -> np.ndarray:
    """Run ``call(start, count, ptr)`` over chunks of ``out`` in threads."""
    n = out.shape[0]
    if n == 0:
        return out
    base = out.ctypes.data
    isz = out.itemsize

    def work(s: int) -> None:
        c = min(_CHUNK, n - s)
        call(s, c, ctypes.c_void_p(base + s * isz))

    starts = range(0, n, _CHUNK)
    if n <= _CHUNK:
        work(0)
    else:
        workers = max(1, min(16, os.cpu_count() or 1))
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, starts))
    return out


def _out(n, dtype, out):
    if out is None:
        return np.empty(n, dtype=dtype)
    if out.dtype != dtype or not out.flags.c_contiguous or out.shape[0] != n:
        raise ValueError("inputs: `out` must be a contiguous array of the requested dtype/length")
    return out


def uniform_int(n: int, lo: int, hi: int, seed: int, dtype=np.int32, out=None) -> np.ndarray:
    """i.i.d. integers uniform in the closed range [lo, hi]."""
    dtype = np.dtype(dtype)
    span = hi - lo + 1
    if span <= 0 or span > (1 << 32):
        raise ValueError("uniform_int: span must be in [1, 2^32]")
    out = _out(n, dtype, out)
    lib, key = _load(), seed_key(seed)
    fn = {np.dtype(np.int32): lib.gen_uniform_i32, np.dtype(np.int64): lib.gen_uniform_i64}[dtype]
    return _fill(out, lambda s, c, p: fn(key, s, c, lo, span, p))


def bernoulli_half(n: int, seed: int, dtype=np.int32, out=None) -> np.ndarray:
    """i.i.d. Bernoulli(1/2) values in {0, 1} (a 0/1 flag array)."""
    dtype = np.dtype(dtype)
    if dtype not in (np.dtype(np.int32), np.dtype(np.int64)):
        raise ValueError("bernoulli_half: int32 or int64")
    out = _out(n, dtype, out)
    lib, key = _load(), seed_key(seed)
    return _fill(out, lambda s, c, p: lib.gen_bernoulli(key, s, c, dtype.itemsize, p))


def uniform_f32(n: int, seed: int, out=None) -> np.ndarray:
    """i.i.d. fp32 values uniform on the grid k * 2^-23 - 1 in [-1, 1)."""
    out = _out(n, np.dtype(np.float32), out)
    lib, key = _load(), seed_key(seed)
    return _fill(out, lambda s, c, p: lib.gen_uniform_f32(key, s, c, p))


def full_range_i32(n: int, seed: int, out=None) -> np.ndarray:
    """i.i.d. int32 uniform over [-2^31, 2^31): the low 32 bits of the hash."""
    out = _out(n, np.dtype(np.int32), out)
    lib, key = _load(), seed_key(seed)
    return _fill(out, lambda s, c, p: lib.gen_full_i32(key, s, c, p))


def hashes(n: int, seed: int, start: int = 0) -> np.ndarray:
    """The raw 64-bit hashes from the C fill (for spot checks)."""
    out = np.empty(n, dtype=np.uint64)
    lib, key = _load(), seed_key(seed)
    return _fill(out, lambda s, c, p: lib.gen_hash_u64(key, start + s, c, p))


def run_keys(n: int, mean_len: int, seed: int, dtype=np.int32) -> np.ndarray:
    """Keys in runs: run lengths i.i.d. uniform in [1, 2*mean_len - 1] (mean
    ``mean_len``), each run's key an i.i.d. draw of the dtype (full-range
    int32, 64-bit hash, or fp32 uniform on the [-1, 1) grid), truncated to n.
    Neighbouring runs share a key only when two draws collide, which merges
    them into one run."""
    dtype = np.dtype(dtype)
    if mean_len < 1:
        raise ValueError("run_keys: mean_len >= 1")
    if n == 0:
        return np.empty(0, dtype=dtype)
    m = -(-n * 11 // (10 * mean_len)) + 1024          # 10% more runs than needed, on average
    lens = uniform_int(m, 1, 2 * mean_len - 1, seed, dtype=np.int64)
    if int(lens.sum()) < n:
        raise RuntimeError("run_keys: drew too few runs")   # far outside the length distribution
    if dtype == np.dtype(np.int32):
        vals = full_range_i32(m, seed + 1)
    elif dtype == np.dtype(np.int64):
        vals = hashes(m, seed + 1).view(np.int64)
    elif dtype == np.dtype(np.float32):
        vals = uniform_f32(m, seed + 1)
    else:
        raise ValueError("run_keys: int32, int64 or float32")
    return np.repeat(vals, lens)[:n]
