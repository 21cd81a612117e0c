"""GB300-native split-K flash-decoding attention.

The compute path is the C-ABI library ``libattn.so`` (hand-written sm_103a
CUDA kernels, declared in ``include/attn_decode.h``).  ``attn`` is its thin
Python binding; submodules are imported lazily so that ``workloads`` (seeded
inputs) can be used without the library.
"""
import importlib

__all__ = ["attn", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
