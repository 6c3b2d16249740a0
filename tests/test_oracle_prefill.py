"""Pins of the chunked-prefill oracle (oracle.prefill_attn).

The prefill oracle evaluates each chunk query row with the single-row decode
oracle over rows [0, cache_index + t].  It is pinned against the uncached
matrix-form causal attention of oracle/causal.py, written separately: the
chunk's outputs must equal rows [c, c + T_new) of full causal attention over
prefix + chunk ("KV-Cache Mechanics", Disabling the Cache: caching does not
change the result; "10.3", section 3: prefill fills the cache for the
prompt's positions).  Planted mistakes in a copy of the oracle -- an
off-by-one causal limit, no mask inside the chunk, interleaved head grouping
-- must each break the pin.
"""
import numpy as np
import pytest

import oracle
from oracle import causal_attention, prefill_attn, widen
from static_kv_cache_gb300 import synth


def _case(B, H, H_kv, d, prefix, T, dtype, seed):
    gen = np.random.default_rng(seed)
    ctx = int(max(prefix)) + T + 3
    def draw(shape):
        x = gen.standard_normal(shape).astype(np.float32)
        if dtype == "fp32":
            return x
        if dtype == "bf16":
            u = x.view(np.uint32)
            return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
        return x.astype(np.float16).view(np.uint16)
    K = draw((B, H_kv, ctx, d))
    V = draw((B, H_kv, ctx, d))
    Q = draw((B, H, ctx, d))           # queries for every position of the full sequence
    return Q, K, V, ctx


def _full_causal_rows(Q, K, V, b, c, T, dtype):
    """Rows [c, c + T) of uncached causal attention over positions [0, c + T)."""
    n = c + T
    Qf = widen(Q[b, :, :n, :], dtype).transpose(1, 0, 2)   # [n, H, d]
    Kf = widen(K[b, :, :n, :], dtype).transpose(1, 0, 2)   # [n, H_kv, d]
    Vf = widen(V[b, :, :n, :], dtype).transpose(1, 0, 2)
    return causal_attention(Qf, Kf, Vf)[c:n].transpose(1, 0, 2)   # [H, T, d]


CASES = [
    # B, H, H_kv, d, prefix per sequence, T_new, dtype
    (2, 4, 4, 16, [0, 5], 7, "fp32"),
    (3, 8, 2, 32, [0, 9, 20], 12, "bf16"),
    (1, 6, 2, 8, [31], 1, "fp16"),
    (2, 8, 1, 16, [3, 0], 16, "fp32"),
]


def _check_against_full(fn, case):
    B, H, H_kv, d, prefix, T, dtype = case
    Q, K, V, ctx = _case(B, H, H_kv, d, prefix, T, dtype, seed=sum(prefix) + T + d)
    ci = np.array(prefix, dtype=np.int64)
    q = np.stack([Q[b, :, prefix[b]:prefix[b] + T, :] for b in range(B)])
    got = fn(q, K, V, ci, T, dtype)
    worst = 0.0
    for b in range(B):
        ref = _full_causal_rows(Q, K, V, b, prefix[b], T, dtype)
        worst = max(worst, float(np.abs(got[b] - ref).max()))
    return worst


@pytest.mark.parametrize("case", CASES, ids=[f"{c[6]}_B{c[0]}_H{c[1]}_Hkv{c[2]}_T{c[5]}" for c in CASES])
def test_prefill_oracle_equals_uncached_causal_rows(case):
    assert _check_against_full(prefill_attn, case) < 1e-12


def test_prefill_of_one_row_is_the_decode_oracle():
    B, H, H_kv, d, prefix, T, dtype = 2, 4, 2, 16, [6, 0], 1, "bf16"
    Q, K, V, ctx = _case(B, H, H_kv, d, prefix, T, dtype, seed=7)
    q = np.stack([Q[b, :, prefix[b]:prefix[b] + 1, :] for b in range(B)])
    got = prefill_attn(q, K, V, prefix, 1, dtype)
    ref = oracle.decode_attn(np.ascontiguousarray(q[:, :, 0, :]), K, V, np.array(prefix) + 1, dtype)
    assert np.array_equal(got[:, :, 0, :], ref)


# ---- planted mistakes: copies of the oracle, each with one error ----------
def _mutant_off_by_one(q, K, V, ci, T, dtype):
    out = np.empty(q.shape, dtype=np.float64)
    for t in range(T):
        valid = (np.asarray(ci) + t + (1 if t == 0 else 0)).astype(np.int32)   # the row misses itself
        out[:, :, t, :] = oracle.decode_attn(np.ascontiguousarray(q[:, :, t, :]), K, V, valid, dtype)
    return out


def _mutant_no_mask_in_chunk(q, K, V, ci, T, dtype):
    out = np.empty(q.shape, dtype=np.float64)
    for t in range(T):
        valid = (np.asarray(ci) + T).astype(np.int32)                           # sees the whole chunk
        out[:, :, t, :] = oracle.decode_attn(np.ascontiguousarray(q[:, :, t, :]), K, V, valid, dtype)
    return out


def _mutant_interleaved_heads(q, K, V, ci, T, dtype):
    B, H = q.shape[:2]
    H_kv = K.shape[1]
    g = H // H_kv
    perm = [(h % H_kv) * g + h // H_kv for h in range(H)]    # head h served as if it were perm[h]
    return prefill_attn(np.ascontiguousarray(q[:, perm]), K, V, ci, T, dtype)[:, np.argsort(perm)]


@pytest.mark.parametrize("mutant", [_mutant_off_by_one, _mutant_no_mask_in_chunk, _mutant_interleaved_heads],
                         ids=["off_by_one", "no_mask_in_chunk", "interleaved_heads"])
def test_planted_mistakes_break_the_pin(mutant):
    # a case with GQA, a prefix and a multi-row chunk
    case = (3, 8, 2, 32, [0, 9, 20], 12, "bf16")
    assert _check_against_full(mutant, case) > 1e-3
