"""The seeded input generators against the recipe they state.

Every workload's input comes from prefix_scan_gb300/inputs.py (a C fill in
csrc/inputs_gen.c, threaded in chunks).  These CPU tests pin it:
- the hash stream is SplitMix64: with key 0 it reproduces the generator's
  published first outputs for seed 0;
- the C fill equals the numpy restatement of the same definition at and
  across the fill's chunk boundaries;
- each value map is the closed form of the hash that the module states
  (multiply-shift integers, the top bit, the 2^-23 fp32 grid, the low 32
  bits), checked element by element;
- run lengths of run_keys lie in [1, 2L-1] with mean about L.
"""
from __future__ import annotations

import ctypes

import numpy as np

from prefix_scan_gb300 import inputs

# SplitMix64 seeded with 0: its first five outputs as published with the
# generator's reference code (Steele, Lea & Flood, OOPSLA 2014; also the
# seeding routine of the xoshiro generators).
SPLITMIX64_SEED0 = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC,
                    0x1B39896A51A8749B]


def _c_hashes(key: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    inputs._load().gen_hash_u64(key, start, count, ctypes.c_void_p(out.ctypes.data))
    return out


def test_hash_stream_is_splitmix64():
    assert [int(h) for h in _c_hashes(0, 0, 5)] == SPLITMIX64_SEED0
    assert [int(h) for h in inputs.hash_block(0, 0, 5, key=0)] == SPLITMIX64_SEED0


def test_c_fill_matches_the_numpy_definition_across_chunks():
    n = 2 * inputs._CHUNK + 12345            # three chunks, filled by threads
    seed = 7
    got = inputs.hashes(n, seed)
    for lo, hi in ((0, 300), (inputs._CHUNK - 300, inputs._CHUNK + 300), (n - 300, n)):
        assert np.array_equal(got[lo:hi], inputs.hash_block(seed, lo, hi - lo))
    # and an offset start lands on the same elements
    assert np.array_equal(inputs.hashes(100, seed, start=5000), got[5000:5100])


def test_value_maps_are_the_stated_closed_forms():
    n, seed = 200_003, 11
    h = inputs.hashes(n, seed)
    for lo, hi in ((0, 9), (-100, 100), (0, (1 << 20) - 1), (1, 31)):
        span = np.uint64(hi - lo + 1)
        want = lo + (((h >> np.uint64(32)) * span) >> np.uint64(32)).astype(np.int64)
        got = inputs.uniform_int(n, lo, hi, seed, dtype=np.int64)
        assert np.array_equal(got, want), (lo, hi)
        assert got.min() >= lo and got.max() <= hi
        assert np.array_equal(inputs.uniform_int(n, lo, hi, seed, dtype=np.int32), want.astype(np.int32))
    assert np.array_equal(inputs.bernoulli_half(n, seed), (h >> np.uint64(63)).astype(np.int32))
    f = inputs.uniform_f32(n, seed)
    want_f = ((h >> np.uint64(40)).astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)
    assert np.array_equal(f, want_f)
    assert f.min() >= -1.0 and f.max() < 1.0
    assert np.all((f.astype(np.float64) + 1.0) * 2.0 ** 23 == np.round((f.astype(np.float64) + 1.0) * 2.0 ** 23))
    assert np.array_equal(inputs.full_range_i32(n, seed), (h & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32))


def test_distributions_look_like_their_names():
    n = 1 << 20
    b = inputs.bernoulli_half(n, 3)
    assert abs(b.mean() - 0.5) < 0.005
    u = inputs.uniform_int(n, 0, 9, 1)
    assert set(np.unique(u)) == set(range(10))
    assert abs(u.mean() - 4.5) < 0.02
    f = inputs.uniform_f32(n, 2)
    assert abs(f.mean()) < 0.005 and abs((f.astype(np.float64) ** 2).mean() - 1.0 / 3.0) < 0.005
    x = inputs.full_range_i32(n, 5)
    assert x.min() < -(1 << 30) and x.max() > (1 << 30)


def test_run_lengths():
    n = 1 << 20
    for mean in (1, 16, 256):
        k = inputs.run_keys(n, mean, 11 + mean)
        heads = np.flatnonzero(np.r_[True, k[1:] != k[:-1]])
        lengths = np.diff(np.r_[heads, n])[:-1]           # the last run is cut at n
        assert lengths.min() >= 1
        # neighbouring runs merge only when two 32-bit draws collide
        assert lengths.max() <= 2 * mean - 1 or np.mean(lengths > 2 * mean - 1) < 1e-3
        assert abs(lengths.mean() - mean) < 0.05 * mean + 0.01
