"""int8 KV cache: quantisation on append and the dequantised rows (numpy).

TEST INFRASTRUCTURE ONLY.

"10.3 -- KV cache implementation details", section 4.4 (KV-cache
quantisation): the cache can be stored in lower precision; fp16 -> int8
halves the memory (p = 1 byte per element in the cache-size formula) at a
small quality cost.  The pages do not fix the scheme (the optimisation
note's "kivi-int8" dtype tag names one without defining it).  Reading taken,
the plainest one that quantises each row as it is appended:
  * symmetric, one fp32 scale per cache row (one token of one KV head, d_h
    elements): absmax = max_d |x_d|, scale = absmax / 127;
  * code_d = rint(x_d * (127 / absmax)), round half to even, in [-127, 127];
    a row of zeros gets scale 0 and codes 0;
  * the attention reads x_hat_d = code_d * scale.
A quantised code is an integer decided by floating point, so every step is
taken in fp32 exactly as written above (IEEE division and multiplication,
round to nearest even), the precision the GPU path uses.
"""
from __future__ import annotations

import numpy as np

from .causal import widen


def quantize_rows(x_bits: np.ndarray, dtype: str):
    """x_bits: [..., d] stored elements (bf16/fp16 as uint16 bits, fp32 as
    float32).  Returns (codes int8 [..., d], scales float32 [...])."""
    x = widen(x_bits, dtype).astype(np.float32)            # exact: 16-bit types fit fp32
    absmax = np.abs(x).max(axis=-1)
    f127 = np.float32(127.0)
    scale = (absmax / f127).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = (f127 / absmax).astype(np.float32)
        prod = (x * inv[..., None]).astype(np.float32)
    codes = np.rint(prod)
    codes = np.where(absmax[..., None] > 0, codes, 0.0)
    codes = np.clip(codes, -127, 127).astype(np.int8)
    return codes, scale


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """code * scale in float64 (exact: an int8 times an fp32 fits a double).
    Scales of rows past the live length may hold a signalling-NaN poison;
    their conversion raises the "invalid" flag, which is ignored (those rows
    are never attended)."""
    with np.errstate(invalid="ignore"):
        return codes.astype(np.float64) * scales.astype(np.float64)[..., None]
