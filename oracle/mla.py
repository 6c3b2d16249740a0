"""MLA latent-cache decode attention (fp64).

TEST INFRASTRUCTURE ONLY.

"10.3 -- KV cache implementation details", section 4.3 (Multi-head Latent
Attention): the cache holds one latent vector c of width d_c per token -- one
tensor, not a K and a V -- and each head's keys and values are rebuilt from
it during attention by low-rank up-projections (DeepSeek-V2: d_c = 512 against
16 heads x 128).  "KV-Cache Mechanics" (MHA vs GQA vs MLA): the latent is
decompressed on the fly, and decoding pays an "absorb" overhead.

Readings taken where the pages stop short:
* head h rebuilds its key and value rows as k = W_UK[h] c and v = W_UV[h] c,
  with W_UK[h] and W_UV[h] of shape [d_h, d_c];
* the scores are scaled by 1/sqrt(d_h), the width of the rebuilt key, like
  every other attention on the pages;
* nothing outside the latent is cached (the pages' MLA size formula counts
  the latent alone), so no separate positional key part exists.

``mla_decode_attn`` is the definition written out: rebuild every head's K and
V rows from the live latents, then the single-query attention over them (the
fp64 decode oracle with one KV head per query head).  The absorbed order the
GPU takes -- W_UK folded into the query, attention over the latents, W_UV
applied to the attended latent -- is equal in exact arithmetic; the pins
check this function against that identity, closed forms and brute force.
"""
from __future__ import annotations

import numpy as np

from .causal import widen


def rebuild_kv(C, W_UK, W_UV, dtype: str):
    """Latents C [B, ctx, d_c] and up-projections W_UK, W_UV [H, d_h, d_c]
    (stored elements) -> float64 K, V [B, H, ctx, d_h]: K[b, h, t] =
    W_UK[h] @ C[b, t] and V[b, h, t] = W_UV[h] @ C[b, t]."""
    c = widen(C, dtype)
    wk = widen(W_UK, dtype)
    wv = widen(W_UV, dtype)
    if wk.shape != wv.shape or wk.shape[2] != c.shape[2]:
        raise ValueError("W_UK and W_UV must be [H, d_h, d_c] with the latent's d_c")
    # [B, 1, ctx, d_c] @ [1, H, d_c, d_h] -> [B, H, ctx, d_h]
    K = np.matmul(c[:, None], np.swapaxes(wk, 1, 2)[None])
    V = np.matmul(c[:, None], np.swapaxes(wv, 1, 2)[None])
    return np.ascontiguousarray(K), np.ascontiguousarray(V)


def mla_decode_attn(q, C, W_UK, W_UV, valid_len, dtype: str, decode_attn=None) -> np.ndarray:
    """out[b, h] = softmax_t(q[b, h] . K[b, h, t] / sqrt(d_h)) . V[b, h, t]
    over t < valid_len[b], with K and V rebuilt from the latents.

    q: [B, H, d_h]; C: [B, ctx, d_c]; W_UK, W_UV: [H, d_h, d_c]; bf16/fp16 as
    uint16 bits, fp32 as float32.  Returns float64 [B, H, d_h].
    """
    if decode_attn is None:
        from . import decode_attn
    q = np.asarray(q)
    B, H, d_h = q.shape
    if np.asarray(W_UK).shape[:2] != (H, d_h) or np.asarray(C).shape[0] != B:
        raise ValueError("shape mismatch between q, the latents and the projections")
    ctx = int(np.max(valid_len)) if np.size(valid_len) else 0
    K, V = rebuild_kv(np.asarray(C)[:, :max(ctx, 1)], W_UK, W_UV, dtype)
    return decode_attn(widen(q, dtype), K, V, np.asarray(valid_len, dtype=np.int32), "fp64")
