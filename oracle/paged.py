"""Paged KV cache: the gather through a block table (numpy).

TEST INFRASTRUCTURE ONLY.

"10.3 -- KV cache implementation details", section 7 (cache management
policies), PagedAttention: the cache is allocated in fixed-size blocks
(16 tokens), like virtual-memory pages, and a block table lets physically
non-contiguous blocks be logically contiguous for the model.  Reading taken
(the pages fix the block size and the table, not the layout): per layer one
pool of physical blocks [num_blocks, H_kv, 16, d_h] for K and one for V, and
one table [B, max_blocks] shared by the layers; token p of sequence b lives in
block table[b, p // 16] at slot p % 16.  Attention over a paged cache is the
decode attention over the rows this gather reproduces.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16


def gather(pool: np.ndarray, table: np.ndarray, ctx: int) -> np.ndarray:
    """pool [num_blocks, H_kv, 16, d] (any dtype), table [B, max_blocks]
    int -> dense [B, H_kv, ctx, d] of the logical rows [0, ctx)."""
    B = table.shape[0]
    num_blocks, H_kv, bs, d = pool.shape
    if bs != BLOCK:
        raise ValueError("blocks hold 16 rows")
    out = np.empty((B, H_kv, ctx, d), dtype=pool.dtype)
    for b in range(B):
        for p in range(ctx):
            out[b, :, p, :] = pool[table[b, p // BLOCK], :, p % BLOCK, :]
    return out
