"""GB300-native (sm_103a) chunked affine scan library for the SAMU recurrent mixer
and the real RG-LRU scan.

The compute path lives in the CUDA shared library ``liblrs_gb300.so`` (built
in-tree by ``__graft_entry__.build()``) behind the C ABI declared in
``include/samu.h``.  The Python functions re-exported here only marshal torch
tensors and streams into that ABI; importing this package does not load the
library, so ``synth`` can be used on machines without the extension.
"""
from __future__ import annotations

__all__ = [
    "samu_workspace_bytes", "samu_forward", "samu_backward",
    "rglru_workspace_bytes", "rglru_forward", "rglru_backward",
    "device_status", "library_path",
]


def __getattr__(name):
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
