"""CPU oracle for the static KV-cache decode step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may.  It shares no code with the CUDA path.

Contents
--------
* ``decode_attn``     -- fp64 single-query attention over the cached rows
                         (C, ``kvc_oracle.c``); "10.3 -- KV cache
                         implementation details", section 5, attention bullet.
* ``ListAppendCache`` -- the concatenating cache that the in-place append
                         must reproduce byte for byte ("KV Cache
                         Optimization...", section #2, Before/After).
* ``causal_attention``-- uncached full causal attention ("KV-Cache
                         Mechanics", Disabling the Cache).
* ``quantize_rows``   -- the int8 cache: symmetric per-row codes and fp32
                         scales ("10.3", section 4.4), and the dequantised
                         rows the attention reads.
* ``paged.gather``    -- the logical rows of a paged cache through its block
                         table ("10.3", section 7, PagedAttention).
* ``prefill_attn``    -- chunked-prefill attention: each chunk query row
                         attends over the rows up to its own position
                         ("10.3", section 3; "KV-Cache Mechanics", AR
                         Static KV-Cache).
* ``mla_decode_attn`` -- MLA decode: K and V rebuilt per head from the
                         cached latents by the up-projections, then the
                         single-query attention ("10.3", section 4.3).
* ``kv_cache_bytes`` and friends -- the cache-size formula ("10.3",
                         section 2 boxed formula; section 4.4).
"""
from __future__ import annotations

import ctypes
import time

import numpy as np

from . import build as _build
from .cache import ListAppendCache
from .causal import causal_attention, widen
from .formula import kv_bytes_per_token, kv_cache_bytes, mla_cache_bytes
from .prefill import prefill_attn
from .mla import mla_decode_attn
from .quant import dequantize_rows, quantize_rows
from . import paged

__all__ = ["decode_attn", "prefill_attn", "mla_decode_attn", "quantize_rows", "dequantize_rows", "ListAppendCache",
           "causal_attention", "widen",
           "kv_cache_bytes", "kv_bytes_per_token", "mla_cache_bytes",
           "load_library", "num_threads", "set_num_threads", "DTYPE_CODES"]

DTYPE_CODES = {"bf16": 0, "fp32": 1, "fp16": 2, "fp64": 3}
_STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "fp64": np.float64}

_lib = None


def _bind(lib):
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    vp = ctypes.c_void_p
    lib.kvo_decode_attn.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i64, i32, vp]
    lib.kvo_decode_attn.restype = ctypes.c_int
    lib.kvo_num_threads.restype = ctypes.c_int
    lib.kvo_set_num_threads.argtypes = [ctypes.c_int]
    lib.kvo_widen.argtypes = [vp, i64, ctypes.c_int]
    lib.kvo_widen.restype = ctypes.c_double
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` loads a
    specific build, e.g. a planted-mistake variant, without caching it."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def num_threads() -> int:
    return load_library().kvo_num_threads()


def set_num_threads(n: int) -> None:
    load_library().kvo_set_num_threads(n)


def _storage(a, dtype: str) -> np.ndarray:
    want = _STORAGE[dtype]
    a = np.asarray(a)
    if dtype == "fp16" and a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError(f"{dtype} data must be stored as {np.dtype(want).name}, got {a.dtype}")
    return np.ascontiguousarray(a)


def decode_attn(q, K, V, valid_len, dtype: str, lib=None) -> np.ndarray:
    """softmax(q K^T / sqrt(d_h)) V over rows [0, valid_len[b]) of each
    sequence's KV head; returns float64 [B, H, d_h].

    q: [B, H, d_h]; K, V: [B, H_kv, ctx, d_h]; bf16/fp16 as uint16 bits.
    """
    lib = lib or load_library()
    q = _storage(q, dtype)
    K = _storage(K, dtype)
    V = _storage(V, dtype)
    B, H, d_h = q.shape
    Bk, H_kv, ctx, dk = K.shape
    if Bk != B or dk != d_h or V.shape != K.shape:
        raise ValueError("shape mismatch between q, K and V")
    vl = np.ascontiguousarray(np.asarray(valid_len, dtype=np.int32))
    if vl.shape != (B,):
        raise ValueError("valid_len must have shape [B]")
    out = np.empty((B, H, d_h), dtype=np.float64)
    rc = lib.kvo_decode_attn(q.ctypes.data, K.ctypes.data, V.ctypes.data,
                             vl.ctypes.data, B, H, H_kv, d_h, ctx,
                             DTYPE_CODES[dtype], out.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def timed_decode_attn(q, K, V, valid_len, dtype: str):
    """decode_attn plus its wall time in seconds (for the CPU baseline)."""
    t0 = time.perf_counter()
    out = decode_attn(q, K, V, valid_len, dtype)
    return out, time.perf_counter() - t0
