"""Exact softmax attention for GB300 (sm_103a): Python binding of the C ABI.

The compute runs in hand-written CUDA kernels inside ``libfa.so`` (built in
this directory by ``build.build()``); this package only marshals arguments.
Calls fail loudly when the library is missing: there is no fallback.
"""
from . import accounting  # noqa: F401

__all__ = ["accounting", "ops"]


def __getattr__(name):
    if name == "ops":
        from . import ops
        return ops
    raise AttributeError(name)
