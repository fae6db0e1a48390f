"""GB300-native CSA2 sparse decode attention.

``csa2`` is the ctypes binding of ``libcsa2.so`` (hand-written sm_103a CUDA
kernels behind the C ABI in ``include/csa2.h``); ``workloads`` draws the
seeded synthetic inputs; ``build`` compiles the library in-tree.

The binding is imported lazily so that ``workloads`` can be used without
loading torch or the CUDA library.
"""
import importlib

__all__ = ["csa2", "workloads", "build"]


def __getattr__(name):
    if name in ("csa2", "workloads", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    mod = importlib.import_module(f"{__name__}.csa2")
    if hasattr(mod, name):
        return getattr(mod, name)
    raise AttributeError(name)
