"""KV-cache size formulas, exact integer arithmetic.

TEST INFRASTRUCTURE ONLY (part of the oracle; the product computes the same
quantities in its own C code).

Sources:
* "10.3 -- KV cache implementation details", section 2 (boxed formula)
  and section 4.4 (the same with n_kv_heads): bytes =
  2 * n_layers * n_kv_heads * d_head * n_ctx * B * p.  Section 2 prints
  n_heads; for GQA the stored heads are the KV heads (section 4.2), so the
  KV-head count is used.
* "Key-value cache" lesson record, specs "Payload estimate" and science
  "The cache grows with every retained position": 2 x B x L x T x Hkv x Dh x s,
  and per token per sequence 2 * L * Hkv * Dh * s.
* "KV-Cache Mechanics", Memory Formula: L x 2 x S x H_kv x d_h x bytes.
* "10.3", section 2.2: bytes per token = 2 * n_layers * n_heads * d_head * p.
* "10.3", section 4.3: MLA stores one latent of width d_c, so
  n_layers * d_c * n_ctx * B * p (no factor of two).

p may be fractional (0.5 for int4, "10.3" section 2); Fractions keep the
result exact.
"""
from __future__ import annotations

from fractions import Fraction


def kv_cache_bytes(n_layers: int, n_kv_heads: int, d_head: int, n_ctx: int,
                   batch: int, p) -> int:
    """2 * n_layers * n_kv_heads * d_head * n_ctx * batch * p, exactly."""
    total = 2 * n_layers * n_kv_heads * d_head * n_ctx * batch * Fraction(p)
    if total.denominator != 1:
        raise ValueError("cache size is not a whole number of bytes")
    return int(total)


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, d_head: int, p) -> int:
    """Growth of one sequence's cache per retained position."""
    return kv_cache_bytes(n_layers, n_kv_heads, d_head, 1, 1, p)


def mla_cache_bytes(n_layers: int, d_c: int, n_ctx: int, batch: int, p) -> int:
    """One latent row of width d_c per token and layer, no K/V pair."""
    total = n_layers * d_c * n_ctx * batch * Fraction(p)
    if total.denominator != 1:
        raise ValueError("cache size is not a whole number of bytes")
    return int(total)
