"""GB300-native MXFP8 grouped-matmul-finalize-routing.

The compute path lives in the CUDA library built from ``csrc/`` (a C ABI,
declared in ``include/gmmfr.h``); :mod:`.binding` marshals torch tensors into
that ABI.  Importing this package does not load the library: the binding
loads it on first use and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
