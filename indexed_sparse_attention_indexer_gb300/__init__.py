"""Indexed sparse attention for GB300 (sm_103a): indexer -> Top-K -> sparse MLA.

The compute lives in the C-ABI library ``libdsi.so`` (hand-written CUDA kernels,
declared in ``include/dsi.h``); ``binding`` marshals torch tensors to it.
``workloads`` draws seeded synthetic inputs.  The library is loaded lazily on
the first call, and a missing build raises instead of falling back.
"""
__all__ = ["binding", "workloads"]
