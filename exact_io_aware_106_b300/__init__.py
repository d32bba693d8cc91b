"""Exact IO-aware attention for B300 (sm_103a).

The compute lives in the C-ABI library ``libattn.so`` built from ``csrc/``
(declared in ``include/attn.h``); :mod:`exact_io_aware_106_b300.attn` is the
thin ctypes binding (argument marshalling only).  The binding is imported
lazily so that the seeded input generators in :mod:`.workloads` can be used
without loading the CUDA library.
"""

__all__ = ["attn", "workloads"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
