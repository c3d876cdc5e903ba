"""Stress of the two-word tile descriptor that 8-byte scans publish.

A 32-bit scan packs flag, call number and value in one 64-bit word, read
and written as one single-copy-atomic access: the fence-free descriptor of
"Single-pass Parallel Prefix Scan with Decoupled Look-back" (summary page,
section 4.4, "Fence-free descriptor updates").  An 8-byte value does not fit
beside a flag in 64 bits, so an int64, pair or affine descriptor is two
words, each tagged with the flag and the call number and holding one half
of the value, stored together.  Each word is atomic on its own; a reader
accepts the pair only when both words carry the current call number and the
same flag, and re-polls it otherwise.

These tests put that rule under stress:
  * torn pairs made by hand (one word A and the other P; one word of an
    earlier call; both P of different calls) fed to the look-back alone:
    each must be waited on like an unpublished tile, never read as a value
    built from mixed halves, and a well-formed P nearer than a torn pair
    must settle the look-back without waiting;
  * a torn pair that a copy engine repairs while the look-back polls it
    (the copy itself may land one word at a time);
  * whole scans that publish two-word descriptors (int64, {int32, fp32}
    pairs, affine maps, reduce-by-key and run-length encoding), 100 times
    each at thousands of tiles, every run against the oracle.
"""
from __future__ import annotations

import ctypes
import time

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
A, P = _lib.PS_FLAG_A, _lib.PS_FLAG_P
TIMEOUT = _lib.PS_ERR_LOOKBACK_TIMEOUT
REPEATS = 100


def _words(flag: int, epoch: int, value: int) -> tuple[int, int]:
    """The two 64-bit words of a well-formed int64 descriptor, as the
    library's own host-side encoder writes them."""
    lib = _lib.load()
    v = np.array([value], dtype=np.int64)
    buf = (ctypes.c_uint64 * 2)()
    assert lib.ps_testing_encode_descriptor(_lib.PS_INT64, flag, epoch, v.ctypes.data, buf) == 0
    return int(buf[0]), int(buf[1])


def _slots(pairs: list[tuple[int, int]]) -> torch.Tensor:
    """Device descriptor array: slot k holds the two words pairs[k]."""
    db = _lib.load().ps_testing_descriptor_bytes(_lib.PS_INT64)
    assert db % 8 == 0 and db >= 16
    raw = np.zeros(len(pairs) * db // 8, dtype=np.uint64)
    for k, (w0, w1) in enumerate(pairs):
        raw[k * db // 8] = w0
        raw[k * db // 8 + 1] = w1
    return torch.from_numpy(raw.view(np.uint8)).to(DEV)


def _probe(desc: torch.Tensor, tile: int, epoch: int, max_polls: int, stream=None):
    """Launch the look-back of `tile` alone; returns (result, status)
    tensors without waiting."""
    lib = _lib.load()
    res = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    status = torch.zeros(1, dtype=torch.int64, device=DEV)
    torch.cuda.synchronize()   # both filled before a probe on another stream reads them
    s = (stream or torch.cuda.current_stream(DEV)).cuda_stream
    _lib.check("ps_testing_lookback",
               lib.ps_testing_lookback(_lib.PS_INT64, desc.data_ptr(), tile, epoch, max_polls,
                                       res.data_ptr(), status.data_ptr(), s))
    return res, status


def _lookback(pairs, epoch: int, max_polls: int = 200) -> tuple[int, int]:
    res, status = _probe(_slots(pairs), len(pairs), epoch, max_polls)
    torch.cuda.synchronize()
    return int(res.item()), int(status.item())


# Distinctive halves: a value read from a torn pair would show them.
LO_A, HI_P = 0x5555_5555, 0x7777_7777
E = 41   # the call number the probes run as


def _torn_a_p(epoch: int = E) -> tuple[int, int]:
    # word 0 of an A descriptor, word 1 of a P descriptor, same call
    return _words(A, epoch, LO_A)[0], _words(P, epoch, HI_P << 32)[1]


def _torn_epochs(flag: int) -> tuple[int, int]:
    # word 0 of this call, word 1 of the previous call, same flag
    return _words(flag, E, (HI_P << 32) | LO_A)[0], _words(flag, E - 1, (HI_P << 32) | LO_A)[1]


@pytest.mark.parametrize("torn", ["flag_A_then_P", "epoch_now_then_previous_A", "both_P_epochs_differ"])
def test_torn_pair_nearest_is_waited_on_and_never_read(torn):
    t = {"flag_A_then_P": _torn_a_p(), "epoch_now_then_previous_A": _torn_epochs(A),
         "both_P_epochs_differ": (_words(P, E - 1, 9)[0], _words(P, E, 9)[1])}[torn]
    # tile 0 P (inclusive 10), tile 1 A (3), tile 2 torn: tile 3 looks back
    pairs = [_words(P, E, 10), _words(A, E, 3), t]
    val, st = _lookback(pairs, E)
    # the torn tile reads as unpublished: the bounded wait runs out, and
    # the tile then counts as the identity -- nothing of its halves enters
    assert st == (E << 8) | TIMEOUT, hex(st)
    assert val == 0, hex(val)


def test_well_formed_pair_behind_a_torn_one_does_not_help():
    # the torn pair is nearer than the well-formed P: it must still be waited on
    pairs = [_words(P, E, 1000), _words(A, E, 3), _words(P, E, 1003), _torn_a_p()]
    val, st = _lookback(pairs, E)
    assert st == (E << 8) | TIMEOUT and val == 0


def test_torn_pair_behind_the_nearest_P_is_never_waited_on():
    # a well-formed P nearer than the torn pair ends the look-back at once
    pairs = [_words(P, E, 1000), _torn_a_p(), _torn_epochs(P), _words(P, E, 1 << 40), _words(A, E, 7)]
    val, st = _lookback(pairs, E, max_polls=1 << 20)
    assert st == 0 and val == (1 << 40) + 7


def test_well_formed_values_with_full_64_bit_halves():
    # both halves of every value in use, carries across the 32-bit boundary
    vals = [0xFFFF_FFFF, 0x1_0000_0001, 0x7FFF_FFFF_FFFF_FFFF, 0xDEAD_BEEF_0000_0001]
    pairs = [_words(P, E, vals[0])] + [_words(A, E, v - (1 << 64) if v >= 1 << 63 else v) for v in vals[1:]]
    val, st = _lookback(pairs, E, max_polls=1 << 20)
    want = sum(vals) % (1 << 64)
    assert st == 0 and (val % (1 << 64)) == want


def test_torn_pair_repaired_while_the_look_back_polls():
    # The look-back of tile 2 polls a torn pair at tile 1 (word 0 of an A,
    # word 1 of a P) on one stream; a copy engine then writes the
    # well-formed P over it from pinned host memory on another stream.  The
    # copy may land one word at a time, so the reader can meet further torn
    # states on the way; it must return exactly the P's value.
    good = _words(P, E, (0x1234 << 32) | 0x9876)
    desc = _slots([_words(P, E, 5), _torn_a_p()])
    db = _lib.load().ps_testing_descriptor_bytes(_lib.PS_INT64)
    fix = torch.from_numpy(np.array(good, dtype=np.uint64).view(np.uint8).copy()).pin_memory()
    poll_stream, copy_stream = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    torch.cuda.synchronize()
    res, status = _probe(desc, 2, E, max_polls=1 << 21, stream=poll_stream)   # bounded: about a second
    time.sleep(0.05)                        # let the probe start polling the torn pair
    with torch.cuda.stream(copy_stream):
        desc[db:db + 16].copy_(fix, non_blocking=True)
    torch.cuda.synchronize()
    assert status.item() == 0, hex(status.item())
    assert res.item() == (0x1234 << 32) | 0x9876


# ---- whole scans: 100 runs each, thousands of tiles -------------------------

N8 = (1 << 24) + 12345   # 8-byte elements: tiles of 4096, about 4100 tiles


def test_int64_scans_repeated_are_bit_exact():
    x = inputs.hashes(N8, 71).view(np.int64)
    t = torch.from_numpy(x).to(DEV)
    o = torch.empty_like(t)
    ws = api.alloc_workspace(torch.int64, N8, DEV)
    for exclusive in (False, True):
        ref = torch.from_numpy(oracle.exclusive(x) if exclusive else oracle.inclusive(x)).to(DEV)
        for k in range(REPEATS):
            api.scan(t, exclusive=exclusive, out=o, workspace=ws)
            assert torch.equal(o, ref), (exclusive, k)
    assert api.device_status(ws) == 0


def _pairs(n: int, seed: int):
    xi = inputs.full_range_i32(n, seed)
    xf = inputs.uniform_f32(n, seed + 1)
    packed = np.empty((n, 2), dtype=np.int32)
    packed[:, 0] = xi
    packed[:, 1] = xf.view(np.int32)
    return xi, xf, packed


def test_pair_scans_repeated_within_bound():
    xi, xf, packed = _pairs(N8, 72)
    t = torch.from_numpy(packed).to(DEV)
    o = torch.empty_like(t)
    ws = api.alloc_workspace(torch.int64, N8, DEV)
    yi, yf, ya = oracle.scan_pair_i32_f32(xi, xf, False)
    ri = torch.from_numpy(yi).to(DEV)
    rf = torch.from_numpy(yf).to(DEV)
    tol = torch.from_numpy(FP32_REL * ya + FP32_ABS).to(DEV)
    for k in range(REPEATS):
        api.scan_pairs(t, out=o, workspace=ws)
        assert torch.equal(o[:, 0], ri), k
        err = (o[:, 1].view(torch.float32).double() - rf).abs()
        assert bool((err <= tol).all()), k
    assert api.device_status(ws) == 0


def test_affine_scans_repeated_within_bound():
    a, b = inputs.uniform_f32(N8, 73), inputs.uniform_f32(N8, 74)
    t = torch.from_numpy(np.stack([a, b], axis=1)).to(DEV)
    o = torch.empty_like(t)
    ws = api.alloc_workspace(torch.int64, N8, DEV)
    A_, B_, Aa, Ba = oracle.scan_affine_f32(a, b, False)
    rA, rB = torch.from_numpy(A_).to(DEV), torch.from_numpy(B_).to(DEV)
    tA = torch.from_numpy(FP32_REL * Aa + FP32_ABS).to(DEV)
    tB = torch.from_numpy(FP32_REL * Ba + FP32_ABS).to(DEV)
    for k in range(REPEATS):
        api.scan_affine(t, out=o, workspace=ws)
        assert bool(((o[:, 0].double() - rA).abs() <= tA).all()), k
        assert bool(((o[:, 1].double() - rB).abs() <= tB).all()), k
    assert api.device_status(ws) == 0


def test_reduce_by_key_and_rle_repeated_are_bit_exact():
    # (run count, value) pairs travel in the same two-word descriptors
    n = (1 << 23) + 333
    keys = inputs.run_keys(n, 16, 75)
    vals = inputs.full_range_i32(n, 76)
    want_k, want_v = oracle.reduce_by_key(keys, vals)
    _, want_c = oracle.reduce_by_key(keys, None)
    m = want_k.shape[0]
    kt, vt = torch.from_numpy(keys).to(DEV), torch.from_numpy(vals).to(DEV)
    uk, agg = torch.empty_like(kt), torch.empty_like(vt)
    nr = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.zeros(api.reduce_by_key_workspace_size(torch.int32, n), dtype=torch.uint8, device=DEV)
    rk, rv = torch.from_numpy(want_k).to(DEV), torch.from_numpy(want_v).to(DEV)
    rc = torch.from_numpy(np.asarray(want_c, dtype=np.int32)).to(DEV)
    for k in range(REPEATS):
        api.reduce_by_key(kt, vt, unique_keys=uk, aggregates=agg, workspace=ws, num_runs=nr)
        assert int(nr.item()) == m and torch.equal(uk[:m], rk) and torch.equal(agg[:m], rv), k
        api.run_length_encode(kt, unique_keys=uk, counts=agg, workspace=ws, num_runs=nr)
        assert int(nr.item()) == m and torch.equal(uk[:m], rk) and torch.equal(agg[:m], rc), k
    assert api.device_status(ws) == 0
