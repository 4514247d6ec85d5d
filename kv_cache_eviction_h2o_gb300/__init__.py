"""GB300-native budgeted-KV decode attention with H2O heavy-hitter eviction
and the HashEvict LSH variant.

The compute path is the CUDA library ``libh2o_gb300.so`` (sm_103a) behind the
C ABI declared in ``include/h2o.h``; ``binding`` is the thin ctypes layer with
the same names.  ``workloads`` draws the seeded synthetic inputs.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads", "binding"]


def __getattr__(name):
    if name == "binding":
        import importlib
        return importlib.import_module(__name__ + ".binding")
    raise AttributeError(name)
