"""Paged-KV decode attention for GB300 (sm_103a).

The kernels live in ``libpkv.so`` (built from ``csrc/`` by ``__graft_entry__.build()``)
behind the C ABI declared in ``include/paged_kv.h``.  ``binding`` marshals torch
tensors into those calls; importing it fails loudly when the library is missing.
``workloads`` draws seeded synthetic inputs and needs no GPU.
"""

import importlib

__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
