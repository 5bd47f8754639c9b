"""GB300-native gated linear-recurrence scans: selective SSM, RG-LRU, HGRN2.

The compute path is the CUDA library ``_build/liblrscan.so`` (C ABI in
``include/lrscan.h``); :mod:`.binding` marshals torch tensors to it.  The
binding is imported on first use of one of its names, so the input
generators in :mod:`.workloads` load without the library.
"""
from . import workloads  # noqa: F401  (pure torch, holds no scan arithmetic)

__all__ = ["workloads", "binding", "selective_scan", "rglru_scan", "hgrn2",
           "check_status", "LrError"]


def __getattr__(name):
    import importlib
    if name in ("build", "binding"):
        return importlib.import_module(f"{__name__}.{name}")
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(importlib.import_module(f"{__name__}.binding"), name)
