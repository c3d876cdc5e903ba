"""GPU parity of the single-pass reduce-by-key and run-length encoding
against the CPU oracle.

Unique keys, run counts and int32 run sums / lengths must match bit for bit;
an fp32 run sum must lie within FP32_REL * (sum of |value| over the run) +
FP32_ABS of the oracle's fp64 sum.  All calls go through the C ABI.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from conftest import FP32_ABS, FP32_REL
from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import _lib, api  # noqa: E402

DEV = torch.device("cuda:0")
KEYS = {"int32": np.int32, "int64": np.int64, "float32": np.float32}
TILE = {"int32": 4096, "float32": 4096, "int64": 2048}


def make_values(kind: str, n: int, seed: int):
    if kind == "int32":
        return inputs.full_range_i32(n, seed)
    if kind == "float32":
        return inputs.uniform_f32(n, seed)
    return None   # run-length encoding


def check(keys: np.ndarray, vals, got_k: np.ndarray, got_v: np.ndarray, runs: int) -> None:
    if vals is None or vals.dtype == np.int32:
        ok, ov = oracle.reduce_by_key(keys, vals)
        assert runs == ok.shape[0], (runs, ok.shape[0])
        assert np.array_equal(got_k[:runs].view(ok.dtype), ok)
        bad = np.flatnonzero(got_v[:runs] != ov)
        assert bad.size == 0, f"{bad.size} run values differ, first at {bad[:5]}"
    else:
        ok, ov, oa = oracle.reduce_by_key(keys, vals)
        assert runs == ok.shape[0], (runs, ok.shape[0])
        assert np.array_equal(got_k[:runs].view(ok.dtype), ok)
        err = np.abs(got_v[:runs].astype(np.float64) - ov)
        bad = np.flatnonzero(~(err <= FP32_REL * oa + FP32_ABS))
        assert bad.size == 0, f"{bad.size} fp32 run sums out of bound, first at {bad[:5]}"


def run(keys: np.ndarray, vals, koff: int = 0, voff: int = 0):
    n = keys.shape[0]
    kt = torch.empty(n + koff, dtype=getattr(torch, keys.dtype.name), device=DEV)[koff:]
    kt.copy_(torch.from_numpy(keys))
    if vals is None:
        uk, agg, cnt = api.run_length_encode(kt)
    else:
        vt = torch.empty(n + voff, dtype=getattr(torch, vals.dtype.name), device=DEV)[voff:]
        vt.copy_(torch.from_numpy(vals))
        uk, agg, cnt = api.reduce_by_key(kt, vt)
    return uk.cpu().numpy(), agg.cpu().numpy(), int(cnt.item())


@pytest.mark.parametrize("kdt", list(KEYS))
@pytest.mark.parametrize("vkind", ["int32", "float32", "rle"])
def test_sizes_and_run_lengths(kdt, vkind):
    T = TILE[kdt]
    sizes = [1, 2, 3, 31, 33, 1000, T - 1, T, T + 1, 3 * T + 17, 40 * T + 5, (1 << 20) + 3]
    for k, n in enumerate(sizes):
        for mean in (1, 3, 16, 300, 5000):
            keys = inputs.run_keys(n, mean, 10 * k + mean, KEYS[kdt])
            vals = make_values(vkind, n, 7 + k)
            uk, agg, runs = run(keys, vals)
            check(keys, vals, uk, agg, runs)


@pytest.mark.parametrize("kdt", list(KEYS))
def test_one_run_and_all_distinct(kdt):
    n = 37 * TILE[kdt] + 11
    same = np.full(n, 5, dtype=KEYS[kdt])
    uk, cnt, runs = run(same, None)
    assert runs == 1 and int(cnt[0]) == n and uk[0] == same[0]
    ones = np.ones(n, dtype=np.int32)
    uk, s, runs = run(same, ones)
    assert runs == 1 and int(s[0]) == n
    distinct = np.arange(n).astype(KEYS[kdt])
    vals = inputs.full_range_i32(n, 3)
    uk, agg, runs = run(distinct, vals)
    assert runs == n and np.array_equal(uk, distinct) and np.array_equal(agg, vals)


@pytest.mark.parametrize("kdt", list(KEYS))
def test_runs_across_tile_boundaries(kdt):
    # runs that end exactly at, just before and just after tile boundaries,
    # and runs that span several tiles
    T = TILE[kdt]
    cuts = sorted({0, T - 1, T, T + 1, 2 * T, 3 * T - 1, 5 * T, 5 * T + 1, 9 * T + 100})
    n = 10 * T + 3
    keys = np.zeros(n, dtype=np.int64)
    for j, c in enumerate(cuts):
        keys[c:] = j + 1
    keys = keys.astype(KEYS[kdt])
    for vkind in ("int32", "float32", "rle"):
        vals = make_values(vkind, n, 4)
        uk, agg, runs = run(keys, vals)
        check(keys, vals, uk, agg, runs)


@pytest.mark.parametrize("kdt", list(KEYS))
def test_unaligned_arrays_take_the_global_path(kdt):
    n = 9 * TILE[kdt] + 77
    keys = inputs.run_keys(n, 7, 21, KEYS[kdt])
    for koff, voff in ((1, 0), (0, 1), (1, 3)):
        for vkind in ("int32", "float32"):
            vals = make_values(vkind, n, 5)
            uk, agg, runs = run(keys, vals, koff, voff)
            check(keys, vals, uk, agg, runs)
    uk, agg, runs = run(keys, None, 1)
    check(keys, None, uk, agg, runs)


def test_fp32_keys_compare_as_bits():
    k = np.array([0.0, -0.0, -0.0, np.nan, np.nan, 1.0, 1.0], dtype=np.float32)
    uk, cnt, runs = run(k, None)
    assert runs == 4 and cnt[:4].tolist() == [1, 2, 2, 2]
    assert np.array_equal(uk[:4].view(np.uint32), k[[0, 1, 3, 5]].view(np.uint32))


def test_outputs_beyond_the_runs_untouched_and_empty_input():
    n = 5 * 4096 + 9
    keys = inputs.run_keys(n, 50, 8)
    kt = torch.from_numpy(keys).to(DEV)
    vt = torch.from_numpy(inputs.full_range_i32(n, 9)).to(DEV)
    uk = torch.full((n,), -77, dtype=torch.int32, device=DEV)
    agg = torch.full((n,), -88, dtype=torch.int32, device=DEV)
    _, _, cnt = api.reduce_by_key(kt, vt, unique_keys=uk, aggregates=agg)
    m = int(cnt.item())
    assert bool((uk[m:] == -77).all()) and bool((agg[m:] == -88).all())
    check(keys, vt.cpu().numpy(), uk.cpu().numpy(), agg.cpu().numpy(), m)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    _, _, cnt = api.reduce_by_key(e, e)
    assert int(cnt.item()) == 0
    _, _, cnt = api.run_length_encode(e)
    assert int(cnt.item()) == 0


def test_workspace_shared_with_scans_and_repeated_calls():
    n = (1 << 22) + 5
    ws = torch.zeros(max(api.reduce_by_key_workspace_size(torch.int32, n), api.workspace_size(torch.int32, n)),
                     dtype=torch.uint8, device=DEV)
    keys = inputs.run_keys(n, 16, 31)
    vals = inputs.uniform_f32(n, 32)
    kt, vt = torch.from_numpy(keys).to(DEV), torch.from_numpy(vals).to(DEV)
    x = inputs.full_range_i32(n, 33)
    xt = torch.from_numpy(x).to(DEV)
    for _ in range(5):
        uk, agg, cnt = api.reduce_by_key(kt, vt, workspace=ws)
        check(keys, vals, uk.cpu().numpy(), agg.cpu().numpy(), int(cnt.item()))
        y = api.scan_inclusive(xt, workspace=ws)
        assert np.array_equal(y.cpu().numpy(), oracle.inclusive(x))
        uk, c, cnt = api.run_length_encode(kt, workspace=ws)
        check(keys, None, uk.cpu().numpy(), c.cpu().numpy(), int(cnt.item()))
    assert api.device_status(ws) == _lib.PS_OK


def test_int32_sums_are_identical_across_runs():
    n = (1 << 24) + 333
    keys = inputs.run_keys(n, 1000, 41)
    vals = inputs.full_range_i32(n, 42)
    kt, vt = torch.from_numpy(keys).to(DEV), torch.from_numpy(vals).to(DEV)
    uk0, agg0, c0 = api.reduce_by_key(kt, vt)
    check(keys, vals, uk0.cpu().numpy(), agg0.cpu().numpy(), int(c0.item()))
    for _ in range(20):
        uk, agg, c = api.reduce_by_key(kt, vt)
        assert int(c.item()) == int(c0.item())
        m = int(c.item())
        assert torch.equal(uk[:m], uk0[:m]) and torch.equal(agg[:m], agg0[:m])


@pytest.mark.parametrize("vkind", ["float32", "rle"])
def test_full_size_32m_pairs(vkind):
    # 2^25 {int32 key, fp32 value} pairs in runs of mean length 16, and the
    # run-length encoding of the same keys: every run is compared
    n = 1 << 25
    keys = inputs.run_keys(n, 16, 2025)
    vals = make_values(vkind, n, 2026)
    uk, agg, runs = run(keys, vals)
    check(keys, vals, uk, agg, runs)
    torch.cuda.empty_cache()


RLE_TILE = {"int32": 16384, "float32": 16384, "int64": 8192}   # keys per run-length-encoding tile


@pytest.mark.parametrize("kdt", list(KEYS))
def test_rle_tile_geometry(kdt):
    # run-length encoding has tiles of its own (64 KiB of keys): lengths
    # around them, and runs cut at tile, warp (1/16 tile), lane (32 or 16
    # keys) and row boundaries
    T = RLE_TILE[kdt]
    for k, n in enumerate([T - 1, T, T + 1, 2 * T, 2 * T + 1, 3 * T - 1, 7 * T + 5]):
        for mean in (1, 2, 7, 1024, T):
            keys = inputs.run_keys(n, mean, 500 + 10 * k + mean, KEYS[kdt])
            uk, cnt, runs = run(keys, None)
            check(keys, None, uk, cnt, runs)
    n = 6 * T + 3
    cuts = sorted({0, T // 16 - 1, T // 16, T // 8, T // 32, T // 32 + 1, T // 512, T // 512 + 1,
                   3 * T // 512 - 1, T - 1, T, 2 * T - T // 16, 2 * T + 1, 4 * T - 1, 4 * T, 5 * T + T // 2})
    keys = np.zeros(n, dtype=np.int64)
    for j, c in enumerate(cuts):
        keys[c:] = j + 1
    keys = keys.astype(KEYS[kdt])
    uk, cnt, runs = run(keys, None)
    check(keys, None, uk, cnt, runs)


def test_positions_above_2p31():
    # n > 2^31: run positions and lengths need unsigned 32-bit arithmetic.
    # Keys i // L (built on the device), so run j is key j of length L, the
    # last one shorter; checked against that closed form on the device.
    n, L = (1 << 31) + 12345, 1000
    keys = torch.empty(n, dtype=torch.int32, device=DEV)
    step = 1 << 28
    for s in range(0, n, step):
        e = min(n, s + step)
        keys[s:e] = (torch.arange(s, e, dtype=torch.int64, device=DEV) // L).to(torch.int32)
    m = (n + L - 1) // L
    uk, cnt, nr = api.run_length_encode(keys)
    assert int(nr.item()) == m
    want = torch.arange(m, dtype=torch.int32, device=DEV)
    assert torch.equal(uk[:m], want)
    assert bool((cnt[:m - 1] == L).all()) and int(cnt[m - 1].item()) == n - (m - 1) * L
    del cnt
    ones = torch.ones(n, dtype=torch.int32, device=DEV)
    uk, sums, nr = api.reduce_by_key(keys, ones, unique_keys=uk)
    assert int(nr.item()) == m
    assert torch.equal(uk[:m], want)
    assert bool((sums[:m - 1] == L).all()) and int(sums[m - 1].item()) == n - (m - 1) * L
    del keys, ones, uk, sums, want
    torch.cuda.empty_cache()


def _tiles_with_run_counts(T: int, counts, dtype, tail: int = 0) -> np.ndarray:
    """Keys made tile by tile (T keys each): tile t holds counts[t] runs of
    near-equal length, with keys no other tile uses, so every tile opens
    with a head and has exactly counts[t] of them; then `tail` distinct keys
    (a last, partial tile full of heads)."""
    parts = []
    for t, r in enumerate(counts):
        r = max(1, min(r, T))
        bounds = (np.arange(T) * r) // T          # run index of each key
        parts.append(t * 65536 + bounds)
    parts.append(len(counts) * 65536 + np.arange(tail))
    return np.concatenate(parts).astype(dtype)


@pytest.mark.parametrize("kdt", list(KEYS))
@pytest.mark.parametrize("vkind", ["int32", "float32", "rle"])
def test_sparse_and_dense_tiles_in_one_call(kdt, vkind):
    # The kernels pack a tile's runs into an output buffer that a writer warp
    # writes once the tile's prefix is known, unless the tile has more runs
    # than a buffer holds; those are written by the compute warps one tile
    # late.  Per-tile run counts around every buffer size of the two kernels
    # and key widths, in shuffled order -- so dense tiles follow sparse ones
    # and the reverse, dense tiles come in a row, and one is still pending
    # when the input ends (the partial last tile is all heads).
    T = RLE_TILE[kdt] if vkind == "rle" else TILE[kdt]
    edges = [256, 319, 320, 321, 340, 341, 342, 383, 384, 385, 511, 512, 513, 671, 672, 673, 799, 800, 801,
             1343, 1344, 1345]
    counts = [c for c in edges if c <= T] + [1, 2, 31, T // 2, T - 1, T, T, T]
    rng = np.random.default_rng(17)
    for rep in range(2):
        order = rng.permutation(len(counts))
        keys = _tiles_with_run_counts(T, [counts[i] for i in order], KEYS[kdt], tail=T // 3 + 5)
        vals = make_values(vkind, keys.shape[0], 40 + rep)
        uk, agg, runs = run(keys, vals)
        check(keys, vals, uk, agg, runs)
