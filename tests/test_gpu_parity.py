"""GPU parity: the CUDA scans against the CPU oracle, element by element.

Integers must match bit for bit (wraparound modulo 2^w); fp32 must lie
within FP32_REL * sum|x| + FP32_ABS of the fp64 oracle at every element.
All calls go through the C ABI (ctypes) of libprefixscan.so.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from conftest import fp32_ok, read_golden
from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU hosts, never run there
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import api  # noqa: E402

DEV = torch.device("cuda:0")
DTYPES = {"int32": (np.int32, torch.int32), "int64": (np.int64, torch.int64),
          "float32": (np.float32, torch.float32)}


def make(dtype: str, n: int, seed: int) -> np.ndarray:
    if dtype == "int32":
        return inputs.full_range_i32(n, seed)
    if dtype == "int64":
        return inputs.hashes(n, seed).view(np.int64)
    return inputs.uniform_f32(n, seed)


def check(y: np.ndarray, x: np.ndarray, exclusive: bool) -> None:
    if x.dtype == np.float32:
        ok = fp32_ok(y, x, exclusive)
        bad = np.flatnonzero(~ok)
        assert bad.size == 0, f"{bad.size} fp32 elements out of bound, first at {bad[:5]}"
    else:
        ref = oracle.exclusive(x) if exclusive else oracle.inclusive(x)
        bad = np.flatnonzero(y != ref)
        assert bad.size == 0, f"{bad.size} mismatches, first at {bad[:5]}: {y[bad[:3]]} vs {ref[bad[:3]]}"


def run(x: np.ndarray, exclusive: bool, inplace: bool = False, algo: str = "decoupled") -> np.ndarray:
    t = torch.from_numpy(x).to(DEV)
    y = api.scan(t, exclusive=exclusive, inplace=inplace, algo=algo)
    if inplace:
        assert y.data_ptr() == t.data_ptr()
    return y.cpu().numpy()


def sizes_for(dtype: str) -> list[int]:
    T = api.tile_elements(DTYPES[dtype][1])
    # up to 2 tiles one CTA scans the whole array; above, the look-back kernel
    # (with look-back units of two tiles from a few thousand tiles on: an odd
    # tile count leaves the last unit a tile past the end)
    return [1, 2, 3, 16, 31, 32, 33, 127, 1000, T - 1, T, T + 1, 2 * T - 3, 2 * T, 2 * T + 1,
            5 * T + 17, 33 * T + 5, 65537, (1 << 20) + 3, 1301 * T + 17, 1302 * T]


@pytest.mark.parametrize("dtype", list(DTYPES))
@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
@pytest.mark.parametrize("inplace", [False, True], ids=["oop", "inplace"])
def test_sizes(dtype, exclusive, inplace):
    for k, n in enumerate(sizes_for(dtype)):
        x = make(dtype, n, 1000 + k)
        check(run(x, exclusive, inplace), x, exclusive)


@pytest.mark.parametrize("name", ["p1_hierarchical_example.txt", "p2_coarsening_example.txt"])
@pytest.mark.parametrize("dtype", list(DTYPES))
def test_worked_examples(name, dtype):
    g = read_golden(name)
    x = np.array(g["input"], dtype=DTYPES[dtype][0])
    assert list(run(x, False).astype(np.int64)) == g["output"]
    assert list(run(x, True).astype(np.int64)) == [0] + g["output"][:-1]


def test_empty_is_noop():
    for dtype, (_, tdt) in DTYPES.items():
        t = torch.empty(0, dtype=tdt, device=DEV)
        assert api.scan_inclusive(t).numel() == 0
        assert api.scan_exclusive(t).numel() == 0


@pytest.mark.parametrize("dtype", list(DTYPES))
def test_unaligned_pointers(dtype):
    # offsets of 1..3 elements break 16-byte alignment: the scalar I/O path
    T = api.tile_elements(DTYPES[dtype][1])
    n = 3 * T + 11
    for off in (1, 2, 3):
        x = make(dtype, n + off, 50 + off)
        t = torch.from_numpy(x).to(DEV)[off:]
        o = torch.empty(n + 4, dtype=t.dtype, device=DEV)[off:off + n]
        for excl in (False, True):
            y = api.scan(t, exclusive=excl, out=o).cpu().numpy()
            check(y, x[off:], excl)


@pytest.mark.parametrize("dtype", list(DTYPES))
def test_16_byte_but_not_32_byte_aligned(dtype):
    # 16-byte aligned arrays take the bulk-copy path; an output that is not
    # also 32-byte aligned makes the 8-byte kernels store each lane's pair of
    # vectors with two 16-byte stores instead of one 32-byte store
    T = api.tile_elements(DTYPES[dtype][1])
    n = 5 * T + 37
    off = 16 // np.dtype(DTYPES[dtype][0]).itemsize
    x = make(dtype, n + off, 90)
    base = torch.from_numpy(x).to(DEV)
    assert base.data_ptr() % 32 == 0
    t = base[off:]
    o = torch.empty(n + off, dtype=t.dtype, device=DEV)[off:]
    for excl in (False, True):
        y = api.scan(t, exclusive=excl, out=o).cpu().numpy()
        check(y, x[off:], excl)
    y = api.scan(t, out=t).cpu().numpy()   # in place at the same offset
    check(y, x[off:], False)


@pytest.mark.parametrize("algo", ["reduce_then_scan", "chained"])
@pytest.mark.parametrize("dtype", list(DTYPES))
def test_comparison_paths(algo, dtype):
    T = api.tile_elements(DTYPES[dtype][1])
    for k, n in enumerate([1, 17, T, T + 1, 7 * T + 3, 1 << 20, (1 << 22) + 9]):
        x = make(dtype, n, 300 + k)
        for excl in (False, True):
            check(run(x, excl, algo=algo), x, excl)
        check(run(x.copy(), False, inplace=True, algo=algo), x, False)


@pytest.mark.parametrize("dtype", list(DTYPES))
def test_guard_regions_untouched(dtype):
    # canaries before and after the output catch tail-tile overruns
    T = api.tile_elements(DTYPES[dtype][1])
    tdt = DTYPES[dtype][1]
    for n in (5, T + 1, 4 * T - 1):
        x = make(dtype, n, 77)
        g = 4096
        buf = torch.full((n + 2 * g,), 0x5A, dtype=tdt, device=DEV)
        out = buf[g:g + n]
        api.scan(torch.from_numpy(x).to(DEV), out=out)
        host = buf.cpu().numpy()
        assert np.all(host[:g] == 0x5A) and np.all(host[g + n:] == 0x5A)
        check(host[g:g + n], x, False)


def test_fp32_small_integers_bit_exact():
    # every partial sum stays below 2^24, so any association order is exact
    n = (1 << 20) + 123
    x = inputs.uniform_int(n, 0, 9, 8).astype(np.float32)
    for excl in (False, True):
        y = run(x, excl)
        ref = (oracle.exclusive(x) if excl else oracle.inclusive(x)).astype(np.float32)
        assert np.array_equal(y, ref)


def test_fp32_nan_and_inf_propagate():
    T = api.tile_elements(torch.float32)
    n = 3 * T
    x = np.ones(n, dtype=np.float32)
    x[T + 5] = np.nan
    y = run(x, False)
    assert np.all(y[:T + 5] == np.arange(1, T + 6, dtype=np.float32))
    assert np.all(np.isnan(y[T + 5:]))
    x = np.ones(n, dtype=np.float32)
    x[2 * T - 1] = np.inf
    y = run(x, False)
    assert np.all(np.isinf(y[2 * T - 1:])) and np.all(np.isfinite(y[:2 * T - 1]))


def test_repeated_runs_are_identical_for_integers():
    # many tiles, many look-back interactions: integer results never vary
    n = (1 << 24) + 1001
    x = inputs.full_range_i32(n, 9)
    ref = oracle.inclusive(x)
    t = torch.from_numpy(x).to(DEV)
    o = torch.empty_like(t)
    ws = api.alloc_workspace(torch.int32, n, DEV)
    r = torch.from_numpy(ref).to(DEV)
    for _ in range(50):
        api.scan_inclusive(t, out=o, workspace=ws)
        assert torch.equal(o, r)
    assert api.device_status(ws) == 0


# ---- the look-back alone, on hand-made descriptors ---------------------------

def _desc_array(dtype: str, entries, epoch: int = 0):
    import ctypes
    from prefix_scan_gb300 import _lib
    lib = _lib.load()
    code = api.dtype_code(DTYPES[dtype][1])
    db = lib.ps_testing_descriptor_bytes(code)
    raw = bytearray(db * len(entries))
    for k, (flag, val) in enumerate(entries):
        v = np.array([val], dtype=DTYPES[dtype][0])
        buf = (ctypes.c_char * db)()
        assert lib.ps_testing_encode_descriptor(code, flag, epoch, v.ctypes.data, buf) == 0
        raw[k * db:(k + 1) * db] = bytes(buf)
    return torch.frombuffer(raw, dtype=torch.uint8).to(DEV), code


def _lookback(dtype: str, entries, tile: int, max_polls: int = 1 << 20, epoch: int = 0,
              written_epoch: int | None = None):
    from prefix_scan_gb300 import _lib
    lib = _lib.load()
    desc, code = _desc_array(dtype, entries, epoch if written_epoch is None else written_epoch)
    res = torch.zeros(1, dtype=DTYPES[dtype][1], device=DEV)
    status = torch.zeros(1, dtype=torch.int64, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    _lib.check("ps_testing_lookback",
               lib.ps_testing_lookback(code, desc.data_ptr(), tile, epoch, max_polls, res.data_ptr(),
                                       status.data_ptr(), s))
    torch.cuda.synchronize()
    return res.item(), status.item()


@pytest.mark.parametrize("dtype", list(DTYPES))
def test_lookback_fig6_snapshot(dtype):
    # Eight partitions each summing to 2 (Fig. 6 snapshot): whatever mix of
    # A and P the predecessors show, tile k's exclusive prefix is 2k.
    g = read_golden("fig6_snapshot.txt")
    A, P = 1, 2
    parts = g["partitions"]
    incl = g["inclusive_prefix"]
    patterns = [
        [P] + [A] * (parts - 1),                 # only tile 0 has its prefix
        [P, P, P, P, A, A, A, A],                # processor 3 done (window of 3 predecessors)
        [P] * parts,                             # everything done: stop at tile k-1
        [P, A, P, A, P, A, P, A],
    ]
    for pat in patterns:
        entries = [(f, incl[k] if f == P else 2) for k, f in enumerate(pat)]
        for tile in range(1, parts):
            val, st = _lookback(dtype, entries[:tile], tile)
            assert st == 0 and val == g["exclusive_prefix"][tile], (pat, tile, val)


@pytest.mark.parametrize("dtype", list(DTYPES))
def test_lookback_slides_over_many_windows(dtype):
    # 1000 predecessors with aggregates only: the window slides back 32 at a time
    m = 1000
    entries = [(2, 3)] + [(1, 3)] * (m - 1)
    val, st = _lookback(dtype, entries, m)
    assert st == 0 and val == 3 * m


def test_lookback_wait_runs_out_without_hanging():
    # a predecessor that never publishes: the bounded wait gives up, reports
    # PS_ERR_LOOKBACK_TIMEOUT tagged with the call's epoch, and the kernel
    # returns normally
    entries = [(2, 5), (1, 5), (0, 0), (1, 5)]
    val, st = _lookback("int32", entries, 4, max_polls=200, epoch=77)
    assert st & 0xFF == 5 and st >> 8 == 77
    x = torch.arange(10, dtype=torch.int32, device=DEV)   # context still usable
    assert api.scan_inclusive(x)[-1].item() == 45


def test_lookback_ignores_descriptors_of_other_calls():
    # descriptors written by an earlier call (another epoch) read as "not
    # published": the look-back waits on them like on X and gives up
    entries = [(2, 5), (1, 5), (1, 5)]
    val, st = _lookback("int32", entries, 3, max_polls=200, epoch=9, written_epoch=8)
    assert st & 0xFF == 5 and st >> 8 == 9
    val, st = _lookback("int64", entries, 3, epoch=9, written_epoch=9)
    assert st == 0 and val == 15


def test_deterministic_mode_is_bitwise_reproducible():
    # fp32 sums depend on association; the deterministic mode fixes it
    n = (1 << 24) + 777
    x = inputs.uniform_f32(n, 123)
    t = torch.from_numpy(x).to(DEV)
    first = api.scan(t, algo="deterministic")
    check(first.cpu().numpy(), x, False)
    for _ in range(20):
        again = api.scan(t, algo="deterministic")
        assert torch.equal(again.view(torch.int32), first.view(torch.int32))
    firste = api.scan(t, exclusive=True, algo="deterministic")
    for _ in range(5):
        assert torch.equal(api.scan(t, exclusive=True, algo="deterministic").view(torch.int32),
                           firste.view(torch.int32))
