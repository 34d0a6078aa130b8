"""GB300-native masked attention over a block-sparse BlockMask (sm_103a).

The compute path is the C-ABI library libfa.so (csrc/, declared in include/fa.h). The Python names here
only marshal arguments into that library; importing this package does not load it until first use.
"""
import importlib

__all__ = ["fa", "synth", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
