"""List-append (concatenating) KV cache: the oracle for the in-place append.

TEST INFRASTRUCTURE ONLY.

"KV Cache Optimization: GQA Audit, In-Place Buffers, Persistent Prompts",
section #2: the "Before" cache grows by concatenating the new rows on the
token axis each step; the "After" cache slice-assigns them into a
pre-allocated buffer at [valid, valid + T_new).  The smoke tests on the same
page require both to generate byte-identical output.  This class is the
"Before" form, one Python list of row byte strings per (layer, sequence, KV
head): appending is list extension, and the row position is implied by the
list length.  The in-place write position (cache_index) therefore has to
equal the live length, which this class checks.

Rewind (``cache.rewind(by:)`` in the same page's file map) drops rows from
the end.
"""
from __future__ import annotations

import numpy as np


class ListAppendCache:
    def __init__(self, n_layers: int, batch: int, n_kv_heads: int, row_bytes: int):
        self.n_layers = n_layers
        self.batch = batch
        self.n_kv_heads = n_kv_heads
        self.row_bytes = row_bytes
        self.k = [[[[] for _ in range(n_kv_heads)] for _ in range(batch)]
                  for _ in range(n_layers)]
        self.v = [[[[] for _ in range(n_kv_heads)] for _ in range(batch)]
                  for _ in range(n_layers)]

    def length(self, layer: int, b: int) -> int:
        return len(self.k[layer][b][0])

    def append(self, layer: int, k_new: np.ndarray, v_new: np.ndarray,
               cache_index, t_new: int) -> None:
        """Append rows k_new[b, kv, t, :] for t < t_new.

        k_new, v_new: arrays of shape [B, H_kv, T_new, row_bytes] (uint8) or
        any array that views as such.  cache_index[b] must equal the live
        length of sequence b.
        """
        kb = np.ascontiguousarray(k_new).view(np.uint8).reshape(
            self.batch, self.n_kv_heads, t_new, self.row_bytes)
        vb = np.ascontiguousarray(v_new).view(np.uint8).reshape(
            self.batch, self.n_kv_heads, t_new, self.row_bytes)
        for b in range(self.batch):
            if int(cache_index[b]) != self.length(layer, b):
                raise ValueError(
                    f"sequence {b}: write position {int(cache_index[b])} is not "
                    f"the live length {self.length(layer, b)}")
        for b in range(self.batch):
            for kv in range(self.n_kv_heads):
                for t in range(t_new):
                    self.k[layer][b][kv].append(kb[b, kv, t].tobytes())
                    self.v[layer][b][kv].append(vb[b, kv, t].tobytes())

    def rewind(self, layer: int, b: int, n: int) -> None:
        for kv in range(self.n_kv_heads):
            del self.k[layer][b][kv][len(self.k[layer][b][kv]) - n:]
            del self.v[layer][b][kv][len(self.v[layer][b][kv]) - n:]

    def rows(self, layer: int, b: int, kv: int, which: str = "k") -> bytes:
        """The live rows of one (layer, sequence, KV head), concatenated."""
        src = self.k if which == "k" else self.v
        return b"".join(src[layer][b][kv])

    def dense(self, layer: int, which: str, ctx: int, fill: int = 0) -> np.ndarray:
        """Materialise [B, H_kv, ctx, row_bytes] uint8 with rows past the live
        length set to ``fill`` (for feeding the attention oracle)."""
        out = np.full((self.batch, self.n_kv_heads, ctx, self.row_bytes), fill,
                      dtype=np.uint8)
        src = self.k if which == "k" else self.v
        for b in range(self.batch):
            for kv in range(self.n_kv_heads):
                rows = src[layer][b][kv]
                if rows:
                    out[b, kv, :len(rows)] = np.frombuffer(
                        b"".join(rows), dtype=np.uint8).reshape(len(rows), self.row_bytes)
        return out
