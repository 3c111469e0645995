"""GB300-native decode attention over a paged KV cache.

The compute path is the C-ABI library ``libpadecode.so`` (hand-written
sm_103a CUDA kernels, declared in ``include/pa_decode.h``).  ``binding``
marshals torch tensors to it; ``workloads`` generates seeded inputs.

The binding is imported lazily so that the input generators can be used on a
machine without the compiled library; any call into the binding raises if
the library is missing -- there is no fallback path.
"""
from __future__ import annotations

import importlib

__all__ = ["binding", "workloads", "decode", "decode_host", "workspace_bytes"]


def __getattr__(name):
    if name in ("binding", "workloads"):
        return importlib.import_module(f"{__name__}.{name}")
    if name in ("decode", "decode_host", "workspace_bytes"):
        return getattr(importlib.import_module(f"{__name__}.binding"), name)
    raise AttributeError(name)
