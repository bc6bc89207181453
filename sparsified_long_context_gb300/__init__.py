"""unip: packed / chunked long-context prefill attention with UniPrefill-style
block selection, as hand-written CUDA kernels for GB300 (sm_103a).

The compute path is libunip.so (C ABI declared in include/unip.h);
:mod:`.binding` is a thin ctypes layer with the same function names,
:mod:`.pipeline` owns device buffers for the four-call step and
:mod:`.workloads` draws the seeded synthetic inputs.
"""
__all__ = ["binding", "pipeline", "workloads", "native_build"]
__version__ = "0.1.0"
