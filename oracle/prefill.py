"""Chunked-prefill attention over a static cache (fp64).

TEST INFRASTRUCTURE ONLY.

"KV-Cache Mechanics", AR Static KV-Cache: prefill is one forward pass over
the prompt that fills the pre-allocated cache starting at cache_index 0;
decoding continues at cache_index = T_prompt.  "10.3 -- KV cache
implementation details", section 3: prefill processes the prompt and
populates the cache for positions 1..L_prompt.  The pages leave the mask
implicit.  Reading: causal -- the only mask under which the prompt processed
in one pass, in chunks, or token by token through the decode step gives the
same outputs, which "KV-Cache Mechanics" (Disabling the Cache) requires of
the cache.  So for a chunk of T_new tokens appended at cache_index c, the
query at chunk position t attends over cache rows [0, c + t]: the decode
definition (one query row against the cached rows) with valid = c + t + 1.
That is what this function writes out, one query row at a time, through the
fp64 decode oracle.
"""
from __future__ import annotations

import numpy as np


def prefill_attn(q, K, V, cache_index, T_new: int, dtype: str, decode_attn=None) -> np.ndarray:
    """out[b, h, t, :] = softmax_j(q[b, h, t] . K[b, h//g, j] / sqrt(d)) . V[b, h//g, j]
    over j < cache_index[b] + t + 1.

    q: [B, H, T_new, d] (bf16/fp16 as uint16 bits, fp32 as float32);
    K, V: [B, H_kv, ctx, d].  Returns float64 [B, H, T_new, d].
    """
    if decode_attn is None:
        from . import decode_attn
    q = np.asarray(q)
    B, H, T, d = q.shape
    if T != T_new:
        raise ValueError("q must hold T_new query rows per head")
    ci = np.asarray(cache_index, dtype=np.int64)
    out = np.empty((B, H, T, d), dtype=np.float64)
    for t in range(T):
        valid = (ci + t + 1).astype(np.int32)
        out[:, :, t, :] = decode_attn(np.ascontiguousarray(q[:, :, t, :]), K, V, valid, dtype)
    return out
