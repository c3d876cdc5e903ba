"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the headers declare, sizes workspaces as documented, and
rejects bad arguments before it enqueues anything.
"""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import pytest

from prefix_scan_gb300 import _lib
from prefix_scan_gb300 import build as nvbuild

INCLUDE = Path(__file__).resolve().parents[1] / "include"


@pytest.fixture(scope="module")
def lib():
    if not nvbuild.is_fresh():
        try:
            nvbuild.build()
        except RuntimeError as e:  # pragma: no cover - toolchain missing
            pytest.skip(f"cannot build the CUDA library here: {e}")
    return _lib.load()


def declared_functions() -> set[str]:
    names = set()
    for h in INCLUDE.glob("*.h"):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(ps_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "ps_scan_inclusive_i32" in names and len(names) >= 15
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares exactly what the headers declare
    assert names == set(_lib.SIGNATURES), names ^ set(_lib.SIGNATURES)


def test_no_process_wide_symbols(lib):
    """A function-local static of an externally visible template instance is
    a GNU-unique symbol, which the dynamic linker binds once per process: a
    second copy of the library (a variant build, another plug-in bundling
    it) would then share the first one's per-device launch records and skip
    its own shared-memory opt-in.  The library must export none."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    syms = subprocess.run([nm, "-D", str(nvbuild.LIBRARY)], capture_output=True, text=True, check=True).stdout
    unique = [line for line in syms.splitlines() if " u " in line]
    assert not unique, unique[:5]


def test_workspace_size(lib):
    assert lib.ps_scan_workspace_size(0, 0) == 0
    for code in (0, 1, 2):
        T = lib.ps_tile_elements(code)
        db = lib.ps_testing_descriptor_bytes(code)
        assert T > 0 and T % 32 == 0
        for n in (1, T, T + 1, 1 << 30):
            tiles = -(-n // T)
            need = lib.ps_scan_workspace_size(code, n)
            assert need >= 256 + tiles * db + tiles * 8 and need % 256 == 0
    assert lib.ps_scan_workspace_size(7, 100) == 0


FAKE = 1 << 40  # never dereferenced: every call below fails validation first


@pytest.fixture
def no_device():
    """The calls with made-up addresses run only where no GPU could receive them."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("made-up device addresses are only passed on hosts without a GPU")


def test_argument_errors(lib, no_device):
    ws_need = lib.ps_scan_workspace_size(0, 1000)
    f = lib.ps_scan_inclusive_i32
    assert f(None, None, 0, None, 0, None) == _lib.PS_OK                       # n == 0: no-op
    assert f(None, FAKE, 1000, FAKE + (1 << 20), ws_need, None) == _lib.PS_ERR_INVALID_ARG
    assert f(FAKE, None, 1000, FAKE + (1 << 20), ws_need, None) == _lib.PS_ERR_INVALID_ARG
    assert f(FAKE, FAKE + 8192, 1000, None, ws_need, None) == _lib.PS_ERR_INVALID_ARG
    assert f(FAKE + 2, FAKE + 8192, 1000, FAKE + (1 << 20), ws_need, None) == _lib.PS_ERR_INVALID_ARG
    assert f(FAKE, FAKE + 8192, 1000, FAKE + (1 << 20) + 8, ws_need, None) == _lib.PS_ERR_INVALID_ARG
    assert f(FAKE, FAKE + 8192, 1000, FAKE + (1 << 20), ws_need - 1, None) == \
        _lib.PS_ERR_WORKSPACE_TOO_SMALL
    # partial overlap of in/out, and workspace overlapping the data
    assert f(FAKE, FAKE + 400, 1000, FAKE + (1 << 20), ws_need, None) == _lib.PS_ERR_OVERLAP
    assert f(FAKE, FAKE + 8192, 1000, FAKE + 8192 + 3200, ws_need, None) == _lib.PS_ERR_OVERLAP
    assert f(FAKE, FAKE + 8192, 1000, FAKE + 256, ws_need, None) == _lib.PS_ERR_OVERLAP
    # generic entry: bad enums
    g = lib.ps_scan
    assert g(9, 0, 0, FAKE, FAKE + 8192, 1000, FAKE + (1 << 20), ws_need, None) == _lib.PS_ERR_INVALID_ARG
    assert g(0, 9, 0, FAKE, FAKE + 8192, 1000, FAKE + (1 << 20), ws_need, None) == _lib.PS_ERR_INVALID_ARG
    # int64 misalignment is checked against 8 bytes
    ws64 = lib.ps_scan_workspace_size(1, 1000)
    assert lib.ps_scan_inclusive_i64(FAKE + 4, FAKE + 16384, 1000, FAKE + (1 << 20), ws64, None) == \
        _lib.PS_ERR_INVALID_ARG


def test_host_scan_argument_errors(lib, no_device):
    n = 1000
    need = lib.ps_scan_host_staging_size(0, n)
    ws = lib.ps_scan_workspace_size(0, n)
    assert lib.ps_scan_host_staging_size(0, 0) == 0 and need >= 2 * 4000
    f = lib.ps_scan_host
    H, D = 1 << 41, 1 << 40   # never dereferenced: each call fails validation first
    assert f(0, 0, None, None, 0, None, 0, None, 0, None) == _lib.PS_OK
    assert f(0, 0, None, H, n, D, need, D + (1 << 30), ws, None) == _lib.PS_ERR_INVALID_ARG
    assert f(0, 0, H + 2, H + 8192, n, D, need, D + (1 << 30), ws, None) == _lib.PS_ERR_INVALID_ARG
    assert f(0, 0, H, H + 8192, n, D + 16, need, D + (1 << 30), ws, None) == _lib.PS_ERR_INVALID_ARG
    assert f(0, 0, H, H + 400, n, D, need, D + (1 << 30), ws, None) == _lib.PS_ERR_OVERLAP
    assert f(0, 0, H, H + 8192, n, D, need - 1, D + (1 << 30), ws, None) == _lib.PS_ERR_WORKSPACE_TOO_SMALL
    assert f(0, 0, H, H + 8192, n, D, need, D + (1 << 30), ws - 1, None) == _lib.PS_ERR_WORKSPACE_TOO_SMALL
    assert f(9, 0, H, H + 8192, n, D, need, D + (1 << 30), ws, None) == _lib.PS_ERR_INVALID_ARG


def test_seeded_argument_errors(lib, no_device):
    ws = lib.ps_scan_workspace_size(0, 1000)
    g = lib.ps_scan_seeded
    # a carry inside the input or the workspace, a misaligned carry
    assert g(0, 0, FAKE, FAKE + 8192, 1000, FAKE + 40, None, FAKE + (1 << 20), ws, None) == _lib.PS_ERR_OVERLAP
    assert g(0, 0, FAKE, FAKE + 8192, 1000, None, FAKE + (1 << 20) + 64, FAKE + (1 << 20), ws, None) == \
        _lib.PS_ERR_OVERLAP
    assert g(0, 0, FAKE, FAKE + 8192, 1000, FAKE + (1 << 22) + 2, None, FAKE + (1 << 20), ws, None) == \
        _lib.PS_ERR_INVALID_ARG


def test_status_strings(lib):
    for code, name in [(0, b"PS_OK"), (1, b"PS_ERR_INVALID_ARG"), (2, b"PS_ERR_WORKSPACE_TOO_SMALL"),
                       (3, b"PS_ERR_OVERLAP"), (4, b"PS_ERR_CUDA"), (5, b"PS_ERR_LOOKBACK_TIMEOUT"),
                       (6, b"PS_ERR_WORKSPACE_NOT_INITIALIZED")]:
        assert lib.ps_status_string(code) == name


def test_descriptor_encoding(lib):
    # each 64-bit word: epoch in bits 34..63, flag in bits 32..33, value bits below
    import numpy as np
    buf = (ctypes.c_char * 16)()
    v32 = np.array([-7], dtype=np.int32)
    assert lib.ps_testing_encode_descriptor(0, 2, 12345, v32.ctypes.data, buf) == 0
    w = int(np.frombuffer(bytes(buf)[:8], dtype=np.uint64)[0])
    assert w >> 34 == 12345 and (w >> 32) & 3 == 2 and w & 0xFFFFFFFF == (-7) & 0xFFFFFFFF
    v64 = np.array([-(1 << 40) - 3], dtype=np.int64)
    assert lib.ps_testing_encode_descriptor(1, 1, (1 << 30) - 1, v64.ctypes.data, buf) == 0
    w0, w1 = (int(x) for x in np.frombuffer(bytes(buf), dtype=np.uint64))
    u = int(v64.view(np.uint64)[0])
    assert w0 >> 34 == w1 >> 34 == (1 << 30) - 1 and (w0 >> 32) & 3 == (w1 >> 32) & 3 == 1
    assert (w0 & 0xFFFFFFFF) | ((w1 & 0xFFFFFFFF) << 32) == u
    assert lib.ps_testing_encode_descriptor(0, 3, 0, v32.ctypes.data, buf) == _lib.PS_ERR_INVALID_ARG
    assert lib.ps_testing_encode_descriptor(0, 1, 1 << 30, v32.ctypes.data, buf) == _lib.PS_ERR_INVALID_ARG


def test_python_layer_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    from prefix_scan_gb300 import api
    with pytest.raises(ValueError, match="CUDA"):
        api.scan_inclusive(torch.arange(10, dtype=torch.int32))


def test_reduce_by_key_workspace_size(lib):
    assert lib.ps_reduce_by_key_workspace_size(0, 0) == 0
    assert lib.ps_reduce_by_key_workspace_size(7, 10) == 0
    for code, tile in ((0, 4096), (2, 4096), (1, 2048)):
        for n in (1, tile, tile + 1, 1 << 30):
            need = lib.ps_reduce_by_key_workspace_size(code, n)
            assert need >= 256 + -(-n // tile) * 16 and need % 256 == 0


def test_reduce_by_key_argument_errors(lib, no_device):
    n = 10_000
    ws = lib.ps_reduce_by_key_workspace_size(0, n)
    K, V, UK, AG, W, C = FAKE, FAKE + (1 << 20), FAKE + (2 << 20), FAKE + (3 << 20), FAKE + (4 << 20), FAKE + (5 << 20)
    f = lib.ps_reduce_by_key
    r = lib.ps_run_length_encode
    assert f(0, 0, None, None, None, None, None, 0, None, 0, None) == _lib.PS_OK        # n == 0, no count
    assert f(0, 1, K, V, UK, AG, C, n, W, ws, None) == _lib.PS_ERR_INVALID_ARG         # int64 values
    assert f(9, 0, K, V, UK, AG, C, n, W, ws, None) == _lib.PS_ERR_INVALID_ARG
    assert f(0, 0, K, None, UK, AG, C, n, W, ws, None) == _lib.PS_ERR_INVALID_ARG      # no values
    assert f(0, 0, K + 2, V, UK, AG, C, n, W, ws, None) == _lib.PS_ERR_INVALID_ARG     # misaligned key
    assert f(0, 0, K, V, UK, AG, C + 4, n, W, ws, None) == _lib.PS_ERR_INVALID_ARG     # misaligned count
    assert f(0, 0, K, V, UK, AG, C, 1 << 32, W, ws, None) == _lib.PS_ERR_INVALID_ARG   # n >= 2^32
    assert f(0, 0, K, V, UK, AG, C, n, W, ws - 1, None) == _lib.PS_ERR_WORKSPACE_TOO_SMALL
    assert f(0, 0, K, V, K + 400, AG, C, n, W, ws, None) == _lib.PS_ERR_OVERLAP        # keys out in keys
    assert f(0, 0, K, V, UK, V, C, n, W, ws, None) == _lib.PS_ERR_OVERLAP              # in place values
    assert f(0, 0, K, V, UK, UK + 8, C, n, W, ws, None) == _lib.PS_ERR_OVERLAP         # outputs overlap
    assert f(0, 0, K, V, UK, AG, AG + 64, n, W, ws, None) == _lib.PS_ERR_OVERLAP       # count in output
    assert f(0, 0, K, V, UK, AG, C, n, UK + 1024, ws, None) == _lib.PS_ERR_OVERLAP     # workspace in output
    assert r(0, K, UK, AG, C, n, W, ws - 1, None) == _lib.PS_ERR_WORKSPACE_TOO_SMALL
    assert r(0, K, K, AG, C, n, W, ws, None) == _lib.PS_ERR_OVERLAP
    ws64 = lib.ps_reduce_by_key_workspace_size(1, n)
    assert ws64 > ws
    assert r(1, K + 4, UK, AG, C, n, W, ws64, None) == _lib.PS_ERR_INVALID_ARG         # int64 keys, 4-aligned


def test_pair_scan_argument_errors(lib, no_device):
    n = 10_000
    ws = lib.ps_scan_workspace_size(1, n)   # 8-byte elements use the int64 workspace
    for f in (lib.ps_scan_pair_i32_f32, lib.ps_scan_affine_f32):
        assert f(0, None, None, 0, None, 0, None) == _lib.PS_OK
        assert f(0, FAKE + 4, FAKE + (1 << 20), n, FAKE + (2 << 20), ws, None) == _lib.PS_ERR_INVALID_ARG
        assert f(0, FAKE, FAKE + (1 << 20), n, FAKE + (2 << 20), ws - 1, None) == _lib.PS_ERR_WORKSPACE_TOO_SMALL
        assert f(1, FAKE, FAKE + 800, n, FAKE + (2 << 20), ws, None) == _lib.PS_ERR_OVERLAP
        assert f(0, None, FAKE, n, FAKE + (2 << 20), ws, None) == _lib.PS_ERR_INVALID_ARG


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "prefix_scan.h"
#include "prefix_scan_testing.h"

int main(void) {
    /* host-only calls: no device is touched */
    size_t ws = ps_scan_workspace_size(PS_INT32, 1000000);
    size_t rbk = ps_reduce_by_key_workspace_size(PS_INT64, 1000000);
    size_t tile = ps_tile_elements(PS_FLOAT32);
    ps_status bad = ps_scan_inclusive_i32(NULL, NULL, 5, NULL, 0, NULL);
    ps_status none = ps_scan_exclusive_i64(NULL, NULL, 0, NULL, 0, NULL);
    printf("%zu %zu %zu %d %d %zu %s\n", ws, rbk, tile, (int)bad, (int)none,
           ps_testing_descriptor_bytes(PS_INT64), ps_status_string(PS_ERR_OVERLAP));
    return 0;
}
"""


def test_headers_serve_a_plain_c99_client(lib, tmp_path):
    # The boundary is a C ABI: both headers compile as strict C99 and a C
    # program links against the library and gets the same answers as the
    # binding (host-only calls; no GPU is needed).
    import shutil
    import subprocess
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = Path(nvbuild.LIBRARY).parent
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{INCLUDE}", str(src),
                        "-o", str(exe), f"-L{libdir}", "-lprefixscan", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    ws, rbk, tile, bad, none, db, overlap = r.stdout.split(maxsplit=6)
    assert int(ws) == lib.ps_scan_workspace_size(0, 1000000) > 0
    assert int(rbk) == lib.ps_reduce_by_key_workspace_size(1, 1000000) > 0
    assert int(tile) == lib.ps_tile_elements(2)
    assert int(bad) == 1 and int(none) == 0   # PS_ERR_INVALID_ARG for NULL with n > 0; n == 0 is a no-op
    assert overlap.strip() and int(db) == lib.ps_testing_descriptor_bytes(1)
