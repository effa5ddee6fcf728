"""Paged-KV continuous-batching decode step for GB300 (sm_103a).

The compute lives in ``libpkv.so`` (CUDA kernels + C++ allocator behind the C
ABI in ``include/pkv.h``); :mod:`.binding` marshals torch tensors into it, and
:mod:`.engine` strings the calls into whole decode steps.  Importing this
package does not load the library; the first call into it does, and raises if
the library has not been built (there is no CPU fallback).
"""
__all__ = ["binding", "build", "workloads"]
