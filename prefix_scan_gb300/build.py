"""Builds the CUDA library ``libprefixscan.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked
into ``prefix_scan_gb300/libprefixscan.so`` (git-ignored).  No CMake, no
torch extension machinery: the product is a plain C-ABI shared library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = ROOT / "_build"
LIBRARY = PKG / "libprefixscan.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libprefixscan.so")


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _deps() -> list[Path]:
    return sources() + sorted(CSRC.glob("*.h")) + sorted(CSRC.glob("*.cuh")) + sorted(INCLUDE.glob("*.h"))


def is_fresh() -> bool:
    if not LIBRARY.exists():
        return False
    t = LIBRARY.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _deps())


def _compile_and_link(srcs: list[Path], obj_dir: Path, target: Path, extra: list[str],
                      verbose: bool) -> Path:
    nvcc = nvcc_path()
    obj_dir.mkdir(parents=True, exist_ok=True)

    def compile_one(src: Path) -> tuple[Path, str]:
        obj = obj_dir / (src.stem + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", str(src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = target.with_name(target.name + f".{os.getpid()}.tmp")
    cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *[str(o) for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, target)
    return target


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> Path:
    """Compile and link the library; returns its path (no-op when fresh)."""
    if not force and not ptxas_info and is_fresh():
        return LIBRARY
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    return _compile_and_link(sources(), BUILD_DIR, LIBRARY, extra, verbose or ptxas_info)


# Smallest tile geometry the scan and select kernels accept: four elements
# per thread, so tiles of 1024 elements (256 threads) for every element
# type -- eight times as many tiles, look-backs and descriptor hand-offs per
# byte as the product build.  Run-length encoding runs four compute warps,
# so 16 KiB tiles (four times as many as the product's 64 KiB; the
# workspace holds a descriptor per 4096 keys, so no smaller); reduce-by-key
# keeps its tiles.  The look-back reads two descriptors per lane (a window
# of 64 tiles), so this build also runs the multi-descriptor window fold,
# which must keep sequence order for the non-commutative operators.  The
# allocation-free entry point is left out: its fixed scratch is sized for
# the product geometry.
TINY_TILE_DEFINES = {"PS_ITEMS32": 4, "PS_ITEMS64": 4, "PS_LOOKBACK_K": 2, "PS_RLE_COMPUTE_WARPS": 4}


def build_variant(name: str, defines: dict[str, int], exclude: tuple[str, ...] = ("scan_noalloc.cu",),
                  force: bool = False) -> Path:
    """Build a second copy of the library with other geometry macros, for
    stress tests: ``_build/<name>/libprefixscan_<name>.so`` (not the
    product library).  No-op when it is newer than every source."""
    obj_dir = BUILD_DIR / name
    target = obj_dir / f"libprefixscan_{name}.so"
    if not force and target.exists() and all(p.stat().st_mtime <= target.stat().st_mtime for p in _deps()):
        return target
    srcs = [p for p in sources() if p.name not in exclude]
    extra = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    return _compile_and_link(srcs, obj_dir, target, extra, False)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
