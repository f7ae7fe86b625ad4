"""GB300-native folded multi-branch verification layer (SpecFold).

The compute path lives in the C-ABI library ``libspecfold.so`` (CUDA kernels
for sm_103a); ``binding`` marshals torch tensors into its entry points.  The
binding is imported lazily so that ``synth`` can be used without a GPU.
"""
import importlib

__all__ = ["binding", "synth"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
