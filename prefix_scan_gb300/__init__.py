"""GB300-native device-wide prefix sum (single-pass decoupled look-back).

The compute lives in the C-ABI CUDA library ``libprefixscan.so`` built from
``csrc/`` for sm_103a; :mod:`prefix_scan_gb300.api` wraps it for PyTorch
tensors and :mod:`prefix_scan_gb300._lib` is the raw ctypes binding.  The
library is loaded on first use and a missing build raises.
"""
from ._lib import PrefixScanError  # noqa: F401


def __getattr__(name):
    # torch-dependent wrappers are imported lazily so that the input
    # generators and workloads can be used without touching CUDA.
    if name in ("scan", "scan_inclusive", "scan_exclusive", "workspace_size", "alloc_workspace",
                "device_status", "tile_elements"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
