"""The synthetic workloads the library is tested and measured on.

Each workload is a dtype, a scan kind (inclusive/exclusive), a placement
(out-of-place or in-place), a length and a seeded value distribution from
:mod:`prefix_scan_gb300.inputs`.  The shapes follow the decoupled look-back
paper's experiments (32-bit integers, lengths 2^10 .. 2^30, section A4 of
the paper summary page); the Bernoulli 0/1 workload is the flag array whose
exclusive scan gives stream-compaction offsets (section 4.4, "in-place
compaction behaviour").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import inputs


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str               # "int32" | "int64" | "float32"
    exclusive: bool
    inplace: bool
    n: int
    dist: str                # key into DISTRIBUTIONS
    seed: int
    sweep: tuple = field(default=())   # extra lengths (sweep workloads)

    @property
    def np_dtype(self):
        return np.dtype(self.dtype)

    @property
    def itemsize(self) -> int:
        return self.np_dtype.itemsize

    def make(self, n: int | None = None, out=None) -> np.ndarray:
        return make_input(self.dist, self.dtype, self.n if n is None else n, self.seed, out=out)

    def describe(self) -> str:
        kind = "exclusive" if self.exclusive else "inclusive"
        place = "in-place" if self.inplace else "out-of-place"
        return f"{self.dtype} {kind} sum scan, {place}, n={self.n}, {DIST_TEXT[self.dist]}"


DIST_TEXT = {
    "u0_9": "uniform integers in [0,9]",
    "f_pm1": "fp32 uniform in [-1,1)",
    "bern": "Bernoulli(0.5) in {0,1}",
    "u0_2p20": "uniform integers in [0,2^20)",
    "full32": "uniform int32 in [-2^31,2^31) (wraps)",
}


def make_input(dist: str, dtype: str, n: int, seed: int, out=None) -> np.ndarray:
    dt = np.dtype(dtype)
    if dist == "u0_9":
        return inputs.uniform_int(n, 0, 9, seed, dt, out=out)
    if dist == "f_pm1":
        if dt != np.float32:
            raise ValueError("f_pm1 is an fp32 distribution")
        return inputs.uniform_f32(n, seed, out=out)
    if dist == "bern":
        return inputs.bernoulli_half(n, seed, dt, out=out)
    if dist == "u0_2p20":
        return inputs.uniform_int(n, 0, (1 << 20) - 1, seed, dt, out=out)
    if dist == "full32":
        if dt != np.int32:
            raise ValueError("full32 is an int32 distribution")
        return inputs.full_range_i32(n, seed, out=out)
    raise KeyError(dist)


SMALL_I32 = Workload("i32_incl_2p20", "int32", False, False, 1 << 20, "u0_9", 1)
F32_2P24 = Workload("f32_incl_2p24", "float32", False, False, 1 << 24, "f_pm1", 2)
I32_EXCL_2P28 = Workload("i32_excl_2p28", "int32", True, False, 1 << 28, "bern", 3)
I64_2P29 = Workload("i64_incl_2p29", "int64", False, False, 1 << 29, "u0_2p20", 4)
I32_INPLACE_SWEEP = Workload(
    "i32_incl_inplace_sweep", "int32", False, True, 1 << 30, "full32", 5,
    sweep=(1, 31, 1000, (1 << 16) + 1, 10_000_000, 999_999_937, 1 << 30))

ALL = (SMALL_I32, F32_2P24, I32_EXCL_2P28, I64_2P29, I32_INPLACE_SWEEP)
BY_NAME = {w.name: w for w in ALL}
