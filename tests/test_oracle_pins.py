"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin is a function ``pin_*(lib)`` that raises AssertionError on a
mismatch.  They check the compiled oracle against:
  * the worked examples the pages print (tests/golden/, each cited there);
  * O(n^2) brute force with exact integer / rational arithmetic;
  * closed forms (x = 1, x = i, x = c) and wraparound special cases;
  * invariants (last = total, exclusive = inclusive shifted, differences);
  * numpy's sequential add.accumulate as an independent library routine.
``test_mutants_are_caught`` plants plausible mistakes in a copy of the
oracle's C source and checks that every one of them fails some pin.
"""
from __future__ import annotations

import itertools
import math
import re
import shutil
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import read_golden
from prefix_scan_gb300 import inputs

M32, M64 = 1 << 32, 1 << 64
INT_TYPES = (np.int32, np.int64)


def _wrap(v: int, dtype) -> int:
    bits = np.dtype(dtype).itemsize * 8
    v %= 1 << bits
    return v - (1 << bits) if v >= 1 << (bits - 1) else v


def _brute(x, dtype, exclusive):
    """y[i] = sum_{j<=i} x[j] (or j<i) by direct summation, exact."""
    n = len(x)
    out = []
    for i in range(n):
        hi = i if exclusive else i + 1
        s = sum(int(x[j]) for j in range(hi)) if np.dtype(dtype).kind == "i" else \
            sum((Fraction(float(x[j])) for j in range(hi)), Fraction(0))
        out.append(_wrap(s, dtype) if np.dtype(dtype).kind == "i" else s)
    return out


# ---------------------------------------------------------------- pins ----

def pin_worked_examples(lib):
    for name in ("p1_hierarchical_example.txt", "p2_coarsening_example.txt"):
        g = read_golden(name)
        b = g["block"]
        for dt in (np.int32, np.int64, np.float32):
            x = np.array(g["input"], dtype=dt)
            y = oracle.inclusive(x, lib)
            assert list(np.asarray(y).astype(np.int64)) == g["output"], (name, dt)
            ye = oracle.exclusive(x, lib)
            assert list(np.asarray(ye).astype(np.int64)) == [0] + g["output"][:-1], (name, dt)
            # step 1: block-local scans; step 2: scan of block sums
            for k in range(0, len(x), b):
                loc = oracle.inclusive(x[k:k + b], lib)
                assert list(np.asarray(loc).astype(np.int64)) == g["local"][k:k + b], (name, k)
            sums = np.array([g["local"][k + b - 1] for k in range(0, len(x), b)], dtype=dt)
            assert list(sums.astype(np.int64)) == g["S"]
            assert list(np.asarray(oracle.inclusive(sums, lib)).astype(np.int64)) == g["S_scan"]


def pin_fig6_snapshot(lib):
    g = read_golden("fig6_snapshot.txt")
    parts, psum = g["partitions"], g["partition_sum"]
    rng = np.random.default_rng(6)
    for size in (1, 3, 7, 64):
        chunks = []
        for _ in range(parts):
            c = rng.integers(-5, 6, size=size)
            c[-1] += psum - c.sum()          # each partition sums to 2
            chunks.append(c)
        for dt in (np.int32, np.int64, np.float32):
            x = np.concatenate(chunks).astype(dt)
            inc = np.asarray(oracle.inclusive(x, lib))
            exc = np.asarray(oracle.exclusive(x, lib))
            ends = [inc[(k + 1) * size - 1] for k in range(parts)]
            starts = [exc[k * size] for k in range(parts)]
            assert [int(v) for v in ends] == g["inclusive_prefix"], (size, dt)
            assert [int(v) for v in starts] == g["exclusive_prefix"], (size, dt)


def pin_brute_force_int(lib):
    rng = np.random.default_rng(1234)
    for dt in INT_TYPES:
        info = np.iinfo(dt)
        for n in list(range(0, 65)):
            x = rng.integers(info.min, info.max, size=n, endpoint=True, dtype=dt)
            for exclusive in (False, True):
                y = (oracle.exclusive if exclusive else oracle.inclusive)(x, lib)
                assert [int(v) for v in y] == _brute(x, dt, exclusive), (dt, n, exclusive)


def pin_brute_force_f32(lib):
    """fp64 oracle vs exact rational prefix sums.

    On the [-1,1) grid k*2^-23 every partial sum of <= 64 terms is exact in
    double, so equality is demanded; for arbitrary fp32 values the
    sequential double sum is within (n-1)*2^-53*sum|x| (Higham, Accuracy and
    Stability of Numerical Algorithms, 2nd ed., eq. 4.4).
    """
    for n in range(0, 65):
        x = inputs.uniform_f32(n, 100 + n)
        for exclusive in (False, True):
            y = (oracle.exclusive if exclusive else oracle.inclusive)(x, lib)
            exact = _brute(x, np.float32, exclusive)
            assert [Fraction(float(v)) for v in y] == exact, (n, exclusive)
    rng = np.random.default_rng(99)
    for n in (5, 33, 64):
        x = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))).astype(np.float32)
        for exclusive in (False, True):
            y = (oracle.exclusive if exclusive else oracle.inclusive)(x, lib)
            exact = _brute(x, np.float32, exclusive)
            absx = _brute(np.abs(x), np.float32, exclusive)
            for i in range(n):
                err = abs(Fraction(float(y[i])) - exact[i])
                assert err <= Fraction(max(n - 1, 1), 2 ** 53) * absx[i], (n, i)


def pin_abs_prefix(lib):
    for n in (0, 1, 2, 17, 64):
        x = inputs.uniform_f32(n, 7 + n)
        for exclusive in (False, True):
            a = oracle.abs_prefix(x, exclusive, lib)
            exact = _brute(np.abs(x), np.float32, exclusive)
            assert [Fraction(float(v)) for v in a] == exact, (n, exclusive)
    x = np.array([-1.0, 2.0, -3.0, 0.5], dtype=np.float32)
    assert list(oracle.abs_prefix(x, False, lib)) == [1.0, 3.0, 6.0, 6.5]
    assert list(oracle.abs_prefix(x, True, lib)) == [0.0, 1.0, 3.0, 6.0]


def pin_closed_forms(lib):
    n = 200_003
    i = np.arange(n, dtype=np.int64)
    for dt in INT_TYPES:
        bits = np.dtype(dt).itemsize * 8
        mask = (1 << bits) - 1
        ones = np.ones(n, dtype=dt)
        assert np.array_equal(oracle.inclusive(ones, lib), (i + 1).astype(dt))
        assert np.array_equal(oracle.exclusive(ones, lib), i.astype(dt))
        # x[i] = i  ->  i(i+1)/2 mod 2^w
        iota = i.astype(dt)
        tri = [(k * (k + 1) // 2) & mask for k in (0, 1, 2, n // 2, n - 1)]
        y = oracle.inclusive(iota, lib)
        for k, t in zip((0, 1, 2, n // 2, n - 1), tri):
            assert int(y[k]) & mask == t, (dt, k)
        # x = c (large, wraps many times)  ->  c*(i+1) mod 2^w
        c = (1 << (bits - 2)) + 12345
        y = oracle.inclusive(np.full(n, c, dtype=dt), lib)
        for k in (0, 1, 3, 77, n - 1):
            assert int(y[k]) & mask == (c * (k + 1)) & mask, (dt, k)
        ye = oracle.exclusive(np.full(n, c, dtype=dt), lib)
        for k in (0, 1, 3, 77, n - 1):
            assert int(ye[k]) & mask == (c * k) & mask, (dt, k)
    # fp32 small integers: every partial sum < 2^24 is exact in any order
    x = inputs.uniform_int(n, 0, 9, 11).astype(np.float32)
    y = oracle.inclusive(x, lib)
    assert np.array_equal(y, np.cumsum(x.astype(np.int64)).astype(np.float64))


def pin_wraparound(lib):
    for dt in INT_TYPES:
        info = np.iinfo(dt)
        x = np.array([info.max, 1, -1, info.min, -1], dtype=dt)
        assert list(oracle.inclusive(x, lib)) == [info.max, info.min, info.max, -1, -2]
        assert list(oracle.exclusive(x, lib)) == [0, info.max, info.min, info.max, -1]


def pin_library_crosscheck(lib):
    for dt in INT_TYPES:
        bits = np.dtype(dt).itemsize * 8
        x = (inputs.full_range_i32(1_000_003, 21) if dt == np.int32
             else inputs.hashes(1_000_003, 22).view(np.int64))
        ref = np.add.accumulate(x.astype(np.int64).view(np.uint64), dtype=np.uint64)
        if bits == 32:
            ref = (ref & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32)
        else:
            ref = ref.view(np.int64)
        assert np.array_equal(oracle.inclusive(x, lib), ref)
        short = x[:500]
        acc = [_wrap(v, dt) for v in itertools.accumulate(int(v) for v in short)]
        assert [int(v) for v in oracle.inclusive(short, lib)] == acc
    xf = inputs.uniform_f32(1_000_003, 23)
    # numpy's add.accumulate is a left-to-right running sum (no pairwise split)
    assert np.array_equal(oracle.inclusive(xf, lib), np.add.accumulate(xf.astype(np.float64)))


def pin_invariants(lib):
    n = 1_000_001
    for dt in INT_TYPES:
        mask = (1 << (np.dtype(dt).itemsize * 8)) - 1
        x = (inputs.full_range_i32(n, 31) if dt == np.int32
             else inputs.hashes(n, 32).view(np.int64))
        inc = oracle.inclusive(x, lib)
        exc = oracle.exclusive(x, lib)
        total = int(np.sum(x.astype(np.int64).view(np.uint64), dtype=np.uint64)) & mask
        assert int(inc[-1]) & mask == total
        assert exc[0] == 0 and np.array_equal(exc[1:], inc[:-1])
        d = (inc[1:].astype(np.int64).view(np.uint64) - inc[:-1].astype(np.int64).view(np.uint64))
        xs = x[1:].astype(np.int64).view(np.uint64)
        assert np.array_equal(d & np.uint64(mask), xs & np.uint64(mask))
    b = inputs.bernoulli_half(n, 33)
    yb = oracle.inclusive(b, lib)
    assert np.all(np.diff(yb) >= 0) and yb[-1] == int(b.sum())
    xf = inputs.uniform_f32(n, 34)
    incf, excf = oracle.inclusive(xf, lib), oracle.exclusive(xf, lib)
    assert excf[0] == 0.0 and np.array_equal(excf[1:], incf[:-1])


def pin_degenerate(lib):
    for dt in (np.int32, np.int64, np.float32):
        e = np.zeros(0, dtype=dt)
        assert oracle.inclusive(e, lib).shape == (0,)
        assert oracle.exclusive(e, lib).shape == (0,)
        one = np.array([7], dtype=dt)
        assert list(oracle.inclusive(one, lib)) == [7]
        assert list(oracle.exclusive(one, lib)) == [0]
    x = np.array([1.0, 2.0, np.nan, 4.0, 5.0], dtype=np.float32)
    y = oracle.inclusive(x, lib)
    assert list(y[:2]) == [1.0, 3.0] and np.all(np.isnan(y[2:]))
    ye = oracle.exclusive(x, lib)
    assert list(ye[:3]) == [0.0, 1.0, 3.0] and np.all(np.isnan(ye[3:]))
    x = np.array([1.0, np.inf, 2.0], dtype=np.float32)
    assert list(oracle.inclusive(x, lib)) == [1.0, np.inf, np.inf]


# ---- stream compaction pins ---------------------------------------------------

def _rand_flags(rng, n, p=0.5):
    # nonzero flags of assorted values: only "nonzero" may matter
    f = (rng.random(n) < p).astype(np.uint8)
    return f * rng.integers(1, 256, n, dtype=np.uint8) if n else f


def pin_select_brute_force(lib):
    rng = np.random.default_rng(77)
    for dt in (np.int32, np.int64, np.float32):
        for n in range(0, 65):
            x = rng.integers(-1000, 1000, n).astype(dt)
            f = _rand_flags(rng, n)
            want = [x[i] for i in range(n) if f[i] != 0]
            assert list(oracle.select(x, f, lib)) == want, (dt, n)
            out, k = oracle.partition(x, f, lib)
            rejected = [x[i] for i in range(n) if f[i] == 0]
            assert k == len(want) and list(out[:k]) == want
            assert list(out[k:]) == rejected[::-1], (dt, n)


def pin_select_library_crosscheck(lib):
    rng = np.random.default_rng(78)
    n = 500_003
    for dt in (np.int32, np.int64, np.float32):
        x = inputs.uniform_int(n, -10**6, 10**6, 79).astype(dt)
        f = _rand_flags(rng, n, 0.3)
        m = f != 0
        assert np.array_equal(oracle.select(x, f, lib), x[m])
        out, k = oracle.partition(x, f, lib)
        assert k == int(m.sum())
        assert np.array_equal(out, np.concatenate([x[m], x[~m][::-1]]))


def pin_select_closed_forms(lib):
    n = 100_001
    x = np.arange(n, dtype=np.int64) * 3 - 7
    assert np.array_equal(oracle.select(x, np.ones(n, np.uint8), lib), x)
    assert oracle.select(x, np.zeros(n, np.uint8), lib).shape == (0,)
    every3 = (np.arange(n) % 3 == 0).astype(np.uint8)
    assert np.array_equal(oracle.select(x, every3, lib), x[::3])
    out, k = oracle.partition(x, np.zeros(n, np.uint8), lib)
    assert k == 0 and np.array_equal(out, x[::-1])
    # the partition is a permutation of the input
    f = (x % 7 == 1).astype(np.uint8)
    out, k = oracle.partition(x, f, lib)
    assert np.array_equal(np.sort(out), np.sort(x))
    assert np.array_equal(oracle.select(x, f, lib), out[:k])


def pin_flags_predicates(lib):
    x = inputs.uniform_int(200_001, -50, 50, 80)
    for dt in (np.int32, np.int64, np.float32):
        xd = x.astype(dt)
        assert np.array_equal(oracle.flags(xd, "nonzero", 0, lib), (xd != 0).astype(np.uint8))
        assert np.array_equal(oracle.flags(xd, "greater", 7, lib), (xd > 7).astype(np.uint8))
        assert np.array_equal(oracle.flags(xd, "less", -3, lib), (xd < -3).astype(np.uint8))
    xf = np.array([np.nan, -0.0, 0.0, 1.5, -np.inf], dtype=np.float32)
    assert list(oracle.flags(xf, "nonzero", 0, lib)) == [1, 0, 0, 1, 1]
    assert list(oracle.flags(xf, "greater", 0.0, lib)) == [0, 0, 0, 1, 0]
    assert list(oracle.flags(xf, "less", 0.0, lib)) == [0, 0, 0, 0, 1]
    big = np.array([np.iinfo(np.int64).max, np.iinfo(np.int64).min], dtype=np.int64)
    assert list(oracle.flags(big, "greater", 0, lib)) == [1, 0]


# ---- running max / min pins -----------------------------------------------------

def _ident(op, dt):
    if np.dtype(dt).kind == "f":
        return -np.inf if op == "max" else np.inf
    info = np.iinfo(dt)
    return info.min if op == "max" else info.max


def pin_scan_op_brute_force(lib):
    rng = np.random.default_rng(90)
    for dt in (np.int32, np.int64, np.float32):
        for n in range(0, 65):
            x = rng.integers(-1000, 1000, n).astype(dt)
            for op in ("max", "min"):
                f = max if op == "max" else min
                inc = [f(x[:i + 1]) for i in range(n)]
                exc = [_ident(op, dt)] + inc[:-1] if n else []
                assert list(oracle.scan_op(x, op, False, lib)) == inc, (dt, n, op)
                assert list(oracle.scan_op(x, op, True, lib)) == exc, (dt, n, op)


def pin_scan_op_library_crosscheck(lib):
    n = 300_007
    for dt in (np.int32, np.int64):
        x = inputs.uniform_int(n, -10**9, 10**9, 91).astype(dt)
        assert np.array_equal(oracle.scan_op(x, "max", False, lib), np.maximum.accumulate(x))
        assert np.array_equal(oracle.scan_op(x, "min", False, lib), np.minimum.accumulate(x))
        e = oracle.scan_op(x, "max", True, lib)
        assert e[0] == np.iinfo(dt).min and np.array_equal(e[1:], np.maximum.accumulate(x)[:-1])
    xf = inputs.uniform_f32(n, 92)
    xf[::1013] = np.nan
    for op, ref in (("max", np.fmax), ("min", np.fmin)):
        want = ref.accumulate(np.concatenate([[_ident(op, np.float32)], xf]).astype(np.float32))
        assert np.array_equal(oracle.scan_op(xf, op, False, lib), want[1:])
        assert np.array_equal(oracle.scan_op(xf, op, True, lib), want[:-1])


def pin_scan_op_closed_forms(lib):
    x = np.arange(-500, 500, dtype=np.int64)            # increasing
    assert np.array_equal(oracle.scan_op(x, "max", False, lib), x)
    assert np.all(oracle.scan_op(x, "min", False, lib) == -500)
    neg = np.full(17, -5, dtype=np.int32)               # all negative: identity matters
    assert list(oracle.scan_op(neg, "max", True, lib)) == [np.iinfo(np.int32).min] + [-5] * 16
    nan = np.array([np.nan, np.nan, 2.0, np.nan, 1.0], dtype=np.float32)
    assert list(oracle.scan_op(nan, "max", False, lib)) == [-np.inf, -np.inf, 2.0, 2.0, 2.0]
    assert list(oracle.scan_op(nan, "min", False, lib)) == [np.inf, np.inf, 2.0, 2.0, 1.0]


# ---- reduce-by-key / RLE pins ----------------------------------------------------

def _runs_python(keys, vals):
    out_k, out_v = [], []
    for k, grp in itertools.groupby(zip(keys.tolist() if keys.dtype.kind != "f" else keys.view(np.uint32).tolist(),
                                        vals.tolist()), key=lambda kv: kv[0]):
        out_k.append(k)
        out_v.append(sum(v for _, v in grp))
    return out_k, out_v


def pin_rbk_brute_force(lib):
    rng = np.random.default_rng(95)
    for kdt in (np.int32, np.int64, np.float32):
        for n in range(0, 65):
            keys = np.sort(rng.integers(0, 6, n)).astype(kdt) if n % 2 else rng.integers(0, 3, n).astype(kdt)
            vals = rng.integers(-50, 50, n).astype(np.int32)
            ok, ov = oracle.reduce_by_key(keys, vals, lib)
            pk, pv = _runs_python(keys, vals)
            rawk = ok.view(np.uint32).tolist() if kdt == np.float32 else ok.tolist()
            assert rawk == pk and ov.tolist() == pv, (kdt, n)
            ok2, counts = oracle.reduce_by_key(keys, None, lib)
            assert counts.tolist() == [sum(1 for _ in g) for _, g in itertools.groupby(
                keys.view(np.uint32).tolist() if kdt == np.float32 else keys.tolist())]
            vf = (vals / 8).astype(np.float32)
            okf, ovf, oaf = oracle.reduce_by_key(keys, vf, lib)
            pkf, pvf = _runs_python(keys, vf.astype(np.float64))
            _, paf = _runs_python(keys, np.abs(vf.astype(np.float64)))
            assert np.array_equal(okf, ok) and np.allclose(ovf, pvf, rtol=0, atol=1e-9)
            assert np.allclose(oaf, paf, rtol=0, atol=1e-9)


def pin_rbk_numpy_crosscheck(lib):
    n = 400_003
    keys = np.repeat(inputs.uniform_int(n // 3 + 1, 0, 5, 96), 3)[:n].astype(np.int64)
    vals = inputs.full_range_i32(n, 97)
    heads = np.flatnonzero(np.r_[True, keys[1:] != keys[:-1]])
    ok, ov = oracle.reduce_by_key(keys, vals, lib)
    assert np.array_equal(ok, keys[heads])
    sums = np.add.reduceat(vals.astype(np.int64), heads)
    assert np.array_equal(ov, (sums & 0xFFFFFFFF).astype(np.uint32).view(np.int32))
    _, counts = oracle.reduce_by_key(keys, None, lib)
    assert np.array_equal(counts, np.diff(np.r_[heads, n])) and counts.sum() == n


def pin_rbk_closed_forms(lib):
    n = 10_000
    same = np.full(n, 7, dtype=np.int32)
    ok, ov = oracle.reduce_by_key(same, np.ones(n, np.int32), lib)
    assert ok.tolist() == [7] and ov.tolist() == [n]
    distinct = np.arange(n, dtype=np.int32)
    ok, ov = oracle.reduce_by_key(distinct, distinct, lib)
    assert np.array_equal(ok, distinct) and np.array_equal(ov, distinct)
    # fp32 keys by bits: -0.0 and +0.0 are different keys, equal NaN bit patterns one key
    kf = np.array([0.0, -0.0, -0.0, np.nan, np.nan, 1.0], dtype=np.float32)
    ok, cnt = oracle.reduce_by_key(kf, None, lib)
    assert cnt.tolist() == [1, 2, 2, 1]


# ---- pair-scan pins --------------------------------------------------------------

def pin_pair_fields_match_scalar_scans(lib):
    # each field of the pair scan is the scalar scan of that field (the
    # scalar scans are pinned above, by other code)
    n = 300_007
    xi = inputs.full_range_i32(n, 101)
    xf = inputs.uniform_f32(n, 102)
    for excl in (False, True):
        yi, yf, ya = oracle.scan_pair_i32_f32(xi, xf, excl, lib)
        assert np.array_equal(yi, oracle.exclusive(xi) if excl else oracle.inclusive(xi))
        assert np.array_equal(yf, oracle.exclusive(xf) if excl else oracle.inclusive(xf))
        assert np.array_equal(ya, oracle.abs_prefix(xf, excl))


def pin_affine_closed_forms(lib):
    n = 5000
    b = inputs.uniform_f32(n, 103)
    ones = np.ones(n, dtype=np.float32)
    A, B, Aa, Ba = oracle.scan_affine_f32(ones, b, False, lib)
    assert np.all(A == 1.0) and np.allclose(B, np.cumsum(b.astype(np.float64)), rtol=0, atol=1e-9)
    a = (inputs.uniform_int(n, 1, 99, 104).astype(np.float32) / 64)
    A, B, _, _ = oracle.scan_affine_f32(a, np.zeros(n, np.float32), False, lib)
    assert np.all(B == 0.0)
    logA = np.cumsum(np.log(a.astype(np.float64)))
    ok = np.abs(logA) < 600
    assert np.allclose(np.log(A[ok]), logA[ok], rtol=0, atol=1e-9)
    r = np.float32(0.75)   # a = r, b = 1: B_k = (1 - r^(k+1)) / (1 - r)
    k = np.arange(200)
    A, B, _, _ = oracle.scan_affine_f32(np.full(200, r), np.ones(200, np.float32), False, lib)
    assert np.allclose(B, (1 - 0.75 ** (k + 1)) / 0.25, rtol=1e-12, atol=0)
    assert np.allclose(A, 0.75 ** (k + 1), rtol=1e-12, atol=0)
    # exclusive: the identity map first, then the inclusive result shifted
    Ae, Be, _, _ = oracle.scan_affine_f32(np.full(200, r), np.ones(200, np.float32), True, lib)
    assert Ae[0] == 1.0 and Be[0] == 0.0 and np.array_equal(Ae[1:], A[:-1]) and np.array_equal(Be[1:], B[:-1])


def pin_affine_brute_force_iteration(lib):
    # F_k(x) = A_k x + B_k must equal applying the maps one by one to x
    rng = np.random.default_rng(105)
    a = rng.uniform(-1.5, 1.5, 60).astype(np.float32)
    b = rng.uniform(-1, 1, 60).astype(np.float32)
    A, B, Aa, Ba = oracle.scan_affine_f32(a, b, False, lib)
    for x0 in (0.0, 1.0, -2.5):
        y = x0
        for k in range(60):
            y = float(a[k]) * y + float(b[k])
            assert abs((A[k] * x0 + B[k]) - y) <= 1e-12 * (1 + abs(y))
    # the magnitudes: the same recurrence over |a|, |b|
    assert np.allclose(Ba, oracle.scan_affine_f32(np.abs(a), np.abs(b), False, lib)[1], rtol=1e-15, atol=0)
    assert np.allclose(Aa, np.abs(A), rtol=1e-15, atol=0)


PINS = [pin_worked_examples, pin_fig6_snapshot, pin_brute_force_int, pin_brute_force_f32,
        pin_abs_prefix, pin_closed_forms, pin_wraparound, pin_library_crosscheck,
        pin_invariants, pin_degenerate, pin_select_brute_force, pin_select_library_crosscheck,
        pin_select_closed_forms, pin_flags_predicates, pin_scan_op_brute_force,
        pin_scan_op_library_crosscheck, pin_scan_op_closed_forms, pin_rbk_brute_force,
        pin_rbk_numpy_crosscheck, pin_rbk_closed_forms, pin_pair_fields_match_scalar_scans,
        pin_affine_closed_forms, pin_affine_brute_force_iteration]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


# ------------------------------------------------------------- mutants ----

# (function, original text, planted mistake): each is a plausible slip.
MUTANTS = [
    ("oracle_inclusive_i32", "sum += xu[i];", "sum -= xu[i];"),                 # wrong sign
    ("oracle_inclusive_i32", "for (size_t i = 0;", "for (size_t i = 1;"),        # dropped term
    ("oracle_inclusive_i32", "sum += xu[i];", "sum += xu[i ? i - 1 : 0];"),     # wrong index
    ("oracle_exclusive_i32", "yu[i] = sum;\n        sum += xi;",
     "sum += xi;\n        yu[i] = sum;"),                                        # emit after add
    ("oracle_exclusive_i32", "uint32_t sum = 0u;", "uint32_t sum = 1u;"),        # wrong identity
    ("oracle_inclusive_i64", "uint64_t sum = 0u;", "uint32_t sum = 0u;"),        # narrow accumulator
    ("oracle_exclusive_i64", "sum += xi;", "sum += xi + (i == 3);"),             # stray term
    ("oracle_inclusive_f32", "double sum = 0.0;", "float sum = 0.0f;"),          # fp32 accumulation
    ("oracle_inclusive_f32", "y[i] = sum;", "y[i] = (float)sum;"),               # rounded output
    ("oracle_exclusive_f32", "y[i] = sum;\n        sum += xi;",
     "sum += xi;\n        y[i] = sum - xi;"),                                    # derived by subtraction
    ("oracle_abs_prefix_f32", "xi = -xi;", "xi = xi;"),                          # dropped abs
    ("oracle_abs_prefix_f32", "if (exclusive) {", "if (!exclusive) {"),          # swapped modes
    ("oracle_select_b32", "if (flags[i])", "if (flags[i] & 1)"),                # low bit only
    ("oracle_partition_b64", "out[n - 1 - r++] = x[i];", "out[k + r++] = x[i];"),  # rejected not from the back
    ("oracle_flags_i32", "x[i] > t", "x[i] >= t"),                              # off-by-one predicate
    ("oracle_flags_f32", "x[i] != 0.0f", "x[i] == x[i]"),                       # NaN test instead of nonzero
    ("oracle_scan_op_i32", "int32_t acc = op == 1 ? INT32_MIN : INT32_MAX;",
     "int32_t acc = 0;"),                                                       # wrong identity
    ("oracle_scan_op_i64", "acc = xi > acc ? xi : acc;", "acc = xi < acc ? xi : acc;"),  # max computes min
    ("oracle_scan_op_f32", "acc = op == 1 ? fmaxf(acc, xi) : fminf(acc, xi);",
     "acc = op == 1 ? (acc > xi ? acc : xi) : fminf(acc, xi);"),               # NaN let in
    ("oracle_rbk_b32_i32", "if (i == 0 || keys[i] != keys[i - 1]) {",
     "if (i == 0 || keys[i] < keys[i - 1]) {"),                                  # runs only on descent
    ("oracle_rbk_b64_i32", "        acc += v;\n", "        acc = v;\n"),           # keeps last value
    ("oracle_rbk_b32_f32", "aacc += fabs((double)vals[i]);", "aacc += (double)vals[i];"),  # dropped abs
    ("oracle_scan_pair_i32_f32", "sf += (double)xf[k];", "sf += (double)xi[k];"),            # wrong field
    ("oracle_scan_affine_f32", "B = ak * B + bk;", "B = A * B + bk;"),                        # wrong factor
    ("oracle_scan_affine_f32", "A = ak * A;", "A = ak + A;"),                                 # sum for product
    ("oracle_scan_affine_f32", "Ba = fabs(ak) * Ba + fabs(bk);", "Ba = Ba + fabs(bk);"),      # dropped factor
]


def _function_span(src: str, name: str) -> tuple[int, int]:
    m = re.search(r"\n((?:void|size_t) " + re.escape(name) + r"\([^)]*\)\s*\{)", src)
    assert m, name
    start = m.start(1)
    depth, k = 0, src.index("{", start)
    while True:
        depth += {"{": 1, "}": -1}.get(src[k], 0)
        if depth == 0:
            return start, k + 1
        k += 1


def _run_pins(lib) -> list[str]:
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def test_mutants_are_caught(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = oracle.SOURCE.read_text()
    survivors = []
    for k, (fn, old, new) in enumerate(MUTANTS):
        a, b = _function_span(src, fn)
        body = src[a:b]
        assert old in body, (fn, old)
        mutated = src[:a] + body.replace(old, new, 1) + src[b:]
        c_path = tmp_path / f"mutant{k}.c"
        c_path.write_text(mutated)
        so = oracle.build(force=True, source=c_path, target=tmp_path / f"mutant{k}.so")
        lib = oracle.load(so)
        if not _run_pins(lib):
            survivors.append((fn, new))
    assert not survivors, f"mutants not caught by any pin: {survivors}"


def test_float_error_model_is_sane():
    # guards the bound used in pin_brute_force_f32 against a silly constant
    assert math.isclose(2.0 ** -53, np.finfo(np.float64).eps / 2)
