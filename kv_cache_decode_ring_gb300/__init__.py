"""GB300-native KV-cache decode step: append, split-K decode attention, trim, chunk, INT8 witnesses.

The compute path is the CUDA library ``libkvc.so`` behind the C ABI declared in
``include/kvc.h``; :mod:`kv_cache_decode_ring_gb300.kvc` is its thin ctypes
binding (argument marshalling only).  :mod:`~kv_cache_decode_ring_gb300.workloads`
draws the seeded synthetic inputs.  Importing the package loads nothing; the
binding loads the library on first use and raises if it is missing.
"""

__all__ = ["kvc", "workloads", "build"]


def __getattr__(name):
    if name in ("kvc", "workloads", "build"):
        import importlib
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
