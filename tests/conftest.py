"""Shared test plumbing: the ``gpu`` marker, golden-file reader, tolerances."""
from __future__ import annotations

import sys
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"

# fp32 acceptance bound against the fp64 oracle (per element):
#   |y[i] - y64[i]| <= FP32_REL * sum_{j<=i} |x[j]| + FP32_ABS
# (exclusive: sum over j < i).  The dynamic look-back re-associates the
# additions from run to run, so one bit pattern cannot be demanded (paper
# summary "Single-pass Parallel Prefix Scan with Decoupled Look-back",
# section A6, third conclusion).
FP32_REL = 1e-5
FP32_ABS = 1e-6


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name: str) -> dict:
    """Parse ``key: v v v`` lines of a golden fixture (``#`` = comment)."""
    out = {}
    for line in (GOLDEN / name).read_text(encoding="utf-8").splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, vals = line.partition(":")
        nums = [int(v) for v in vals.split()]
        out[key.strip()] = nums[0] if len(nums) == 1 else nums
    return out


def fp32_ok(y: np.ndarray, x: np.ndarray, exclusive: bool) -> np.ndarray:
    """Per-element mask: fp32 result ``y`` within the bound of the fp64 oracle."""
    import oracle

    ref = oracle.exclusive(x) if exclusive else oracle.inclusive(x)
    a = oracle.abs_prefix(x, exclusive)
    y64 = np.asarray(y, dtype=np.float64)
    ok = np.abs(y64 - ref) <= FP32_REL * a + FP32_ABS
    ok |= np.isnan(y64) & np.isnan(ref)
    ok |= np.isinf(y64) & (y64 == ref)
    return ok


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()
