"""Exact softmax attention for GB300 (sm_103a): Python binding of the C ABI.

The compute runs in hand-written CUDA kernels inside ``libfa.so`` (built in
this directory by ``build.build()``); this package only marshals arguments.
The library is loaded on the first call, and a missing library raises: there
is no fallback.
"""
from . import accounting, ops  # noqa: F401

__all__ = ["accounting", "ops"]
