"""Uncached causal attention in matrix form (numpy, fp64).

TEST INFRASTRUCTURE ONLY.

"KV-Cache Mechanics", Disabling the Cache: generation with the cache off
must give the same tokens.  "10.3 -- KV cache implementation details",
section 2: the keys and values of positions before t never change as t
advances, which is why caching them is exact.  So the decode output at step
t (query q_t over cached rows 0..t) must equal row t of full causal
attention recomputed over all positions at once.  This module is that
recompute: the full T x T score matrix per query head, masked above the
diagonal, a row softmax, then a product with V.  It is written separately
from the single-row oracle in kvc_oracle.c so that one can check the other.
"""
from __future__ import annotations

import numpy as np


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored elements -> float64, exactly.  bf16/fp16 arrive as uint16 bits,
    fp32 as float32.

    Cache rows past a sequence's live length hold the tests' NaN poison,
    whose bit patterns are signalling NaNs; widening one raises the
    floating-point "invalid" flag on some hosts (numpy then warns).  Those
    rows are widened with the rest of a slab but never attended, so the flag
    is ignored here."""
    a = np.asarray(a)
    with np.errstate(invalid="ignore"):
        if dtype == "bf16":
            if a.dtype != np.uint16:
                raise TypeError(f"bf16 data must arrive as uint16 bits, got {a.dtype}")
            return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if dtype == "fp16":
            if a.dtype not in (np.uint16, np.float16):
                raise TypeError(f"fp16 data must arrive as uint16 bits, got {a.dtype}")
            return a.view(np.float16).astype(np.float64)
        if dtype == "fp32":
            if a.dtype != np.float32:
                raise TypeError(f"fp32 data must arrive as float32, got {a.dtype}")
            return a.astype(np.float64)
    raise ValueError(dtype)


def causal_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Q: [T, H, d] ; K, V: [T, H_kv, d] (float64).  Returns [T, H, d].

    Query head h reads KV head h // (H // H_kv) (contiguous grouping).
    """
    T, H, d = Q.shape
    H_kv = K.shape[1]
    g = H // H_kv
    out = np.empty_like(Q)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)      # j > i is the future
    for h in range(H):
        kv = h // g
        S = (Q[:, h, :] @ K[:, kv, :].T) / np.sqrt(d)
        S[mask] = -np.inf
        S = S - S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ V[:, kv, :]
    return out
