"""Fine-grained-scaled FP8 linear layer for GB300 (sm_103a).

The compute path is the CUDA library ``libqlinear.so`` (built from ``csrc/``)
behind a C ABI; ``ops`` is a thin ctypes binding over it. Importing the package
does not load the library; the first op call does, and raises if it is missing.
"""
__all__ = ["ops", "linear", "synthetic"]
