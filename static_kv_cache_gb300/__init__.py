"""Static KV-cache decode for GB300 (sm_103a).

The compute path is ``libkvc.so`` (CUDA kernels behind the C ABI in
``include/kvc.h``); ``static_kv_cache_gb300.kvc`` is its thin ctypes binding
with the same function names.  ``synth`` draws the seeded synthetic inputs.
Importing the binding raises if the library has not been built: there is no
fallback implementation.
"""
__all__ = ["kvc", "synth"]
