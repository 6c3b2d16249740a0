"""Pins of the paged-cache gather (oracle.paged.gather).

"10.3", section 7 (PagedAttention): fixed 16-token blocks, logically
contiguous through a block table.  Pinned by an independent construction --
a dense cache cut into blocks with numpy reshapes and stored under a random
permutation -- which the gather must return exactly; by attention over the
gathered rows equalling attention over the dense rows; and by planted
mistakes (slot and block swapped, the block index off by one).
"""
import numpy as np
import pytest

import oracle
from oracle import paged


def _paged_from_dense(dense, seed):
    """dense [B, H_kv, T, d] (T a multiple of 16) -> (pool, table) with the
    blocks stored at shuffled physical positions."""
    B, H_kv, T, d = dense.shape
    nb = T // 16
    blocks = dense.reshape(B, H_kv, nb, 16, d).transpose(0, 2, 1, 3, 4).reshape(B * nb, H_kv, 16, d)
    perm = np.random.default_rng(seed).permutation(B * nb + 5)[:B * nb]   # spare physical blocks too
    pool = np.zeros((B * nb + 5, H_kv, 16, d), dtype=dense.dtype)
    pool[perm] = blocks
    table = perm.reshape(B, nb)
    return pool, table


def test_gather_returns_the_dense_rows():
    gen = np.random.default_rng(1)
    dense = gen.standard_normal((3, 2, 64, 8)).astype(np.float32)
    pool, table = _paged_from_dense(dense, seed=2)
    assert np.array_equal(paged.gather(pool, table, 64), dense)
    assert np.array_equal(paged.gather(pool, table, 37), dense[:, :, :37])


def test_attention_over_a_paged_cache_equals_the_dense_attention():
    gen = np.random.default_rng(3)
    B, H, H_kv, T, d = 3, 8, 2, 96, 16
    K = gen.standard_normal((B, H_kv, T, d)).astype(np.float32)
    V = gen.standard_normal((B, H_kv, T, d)).astype(np.float32)
    q = gen.standard_normal((B, H, d)).astype(np.float32)
    valid = np.array([96, 17, 40])
    kp, tab = _paged_from_dense(K, seed=4)
    vp = np.zeros_like(kp)
    vp[tab.reshape(-1)] = V.reshape(B, H_kv, T // 16, 16, d).transpose(0, 2, 1, 3, 4).reshape(-1, H_kv, 16, d)
    ref = oracle.decode_attn(q, K, V, valid, "fp32")
    got = oracle.decode_attn(q, paged.gather(kp, tab, T), paged.gather(vp, tab, T), valid, "fp32")
    assert np.array_equal(got, ref)


def _g_slot_block_swapped(pool, table, ctx):
    B = table.shape[0]
    out = np.empty((B, pool.shape[1], ctx, pool.shape[3]), dtype=pool.dtype)
    for b in range(B):
        for p in range(ctx):
            out[b, :, p, :] = pool[table[b, p % 16 % table.shape[1]], :, (p // 16) % 16, :]
    return out


def _g_block_off_by_one(pool, table, ctx):
    B = table.shape[0]
    out = np.empty((B, pool.shape[1], ctx, pool.shape[3]), dtype=pool.dtype)
    for b in range(B):
        for p in range(ctx):
            out[b, :, p, :] = pool[table[b, min((p + 1) // 16, table.shape[1] - 1)], :, p % 16, :]
    return out


@pytest.mark.parametrize("mutant", [_g_slot_block_swapped, _g_block_off_by_one], ids=["slot_block_swapped", "block_off_by_one"])
def test_planted_mistakes_break_the_pin(mutant):
    gen = np.random.default_rng(5)
    dense = gen.standard_normal((2, 2, 64, 8)).astype(np.float32)
    pool, table = _paged_from_dense(dense, seed=6)
    assert not np.array_equal(mutant(pool, table, 64), dense)
