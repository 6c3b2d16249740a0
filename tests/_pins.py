"""Checks that pin the fp64 attention oracle to things other than itself.

Each ``pin_*`` function takes an oracle library handle (the normal build, or
a build with a planted mistake) and raises AssertionError if the oracle
disagrees with the independent reference.  The references are:

* a library routine: ``torch.nn.functional.scaled_dot_product_attention`` in
  fp64 on repeat-interleaved KV heads;
* closed forms: one live row returns that V row exactly; equal keys or a zero
  query return the mean of the V rows; one dominant score returns its V row;
* the cached == uncached invariant ("KV-Cache Mechanics", Disabling the
  Cache; "10.3 -- KV cache implementation details", section 2): decode at
  step t equals row t of full causal attention (``oracle.causal``);
* GQA == MHA on repeated heads ("KV Cache Optimization...", #1 Fix: presets
  with nKvHeads == nHeads keep the old behaviour);
* brute force on tiny inputs with Python floats and ``math.exp``, forming the
  softmax as exp(s) / sum exp(s) without the max shift;
* widening of bf16 / fp16 bits checked against torch's own conversions.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from oracle.causal import widen
from static_kv_cache_gb300 import synth


def _inputs(dtype, B, H, H_kv, d, ctx, seed):
    q = synth.to_bits(synth.normal((B, H, d), dtype, synth.sub_seed(seed, "q")))
    K = synth.to_bits(synth.normal((B, H_kv, ctx, d), dtype, synth.sub_seed(seed, "k")))
    V = synth.to_bits(synth.normal((B, H_kv, ctx, d), dtype, synth.sub_seed(seed, "v")))
    return q, K, V


def _sdpa_reference(q, K, V, valid, dtype, g):
    B, H, d = q.shape
    out = np.empty((B, H, d))
    for b in range(B):
        n = int(valid[b])
        qt = torch.from_numpy(widen(q[b], dtype))[:, None, :]                    # [H, 1, d]
        kt = torch.from_numpy(widen(K[b, :, :n], dtype)).repeat_interleave(g, dim=0)
        vt = torch.from_numpy(widen(V[b, :, :n], dtype)).repeat_interleave(g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
        out[b] = o[:, 0, :].numpy()
    return out


def pin_library_sdpa(lib, dtype="bf16", B=3, H=8, H_kv=2, d=32, ctx=40, seed=7):
    q, K, V = _inputs(dtype, B, H, H_kv, d, ctx, seed)
    valid = np.array([1, 17, ctx][:B] + [ctx] * max(0, B - 3), dtype=np.int32)
    got = oracle.decode_attn(q, K, V, valid, dtype, lib=lib)
    ref = _sdpa_reference(q, K, V, valid, dtype, H // H_kv)
    err = np.abs(got - ref).max()
    assert err < 1e-10, f"oracle vs fp64 SDPA: max abs diff {err}"


def pin_single_row(lib, dtype="bf16"):
    B, H, H_kv, d, ctx = 2, 4, 2, 16, 8
    q, K, V = _inputs(dtype, B, H, H_kv, d, ctx, 11)
    got = oracle.decode_attn(q, K, V, np.ones(B, np.int32), dtype, lib=lib)
    for b in range(B):
        for h in range(H):
            want = widen(V[b, h // (H // H_kv), 0], dtype)
            assert np.array_equal(got[b, h], want), "one live row must return that V row exactly"


def pin_equal_keys_mean(lib, dtype="fp32"):
    B, H, H_kv, d, ctx, n = 1, 2, 1, 8, 12, 9
    q, K, V = _inputs(dtype, B, H, H_kv, d, ctx, 13)
    K[:] = K[:, :, :1, :]                       # every key row equal
    got = oracle.decode_attn(q, K, V, np.array([n], np.int32), dtype, lib=lib)
    want = widen(V[0, 0, :n], dtype).mean(axis=0)
    for h in range(H):
        assert np.abs(got[0, h] - want).max() < 1e-12, "equal keys must give the mean of V"


def pin_zero_query_mean(lib, dtype="bf16"):
    B, H, H_kv, d, ctx, n = 1, 2, 2, 8, 12, 7
    q, K, V = _inputs(dtype, B, H, H_kv, d, ctx, 17)
    q[:] = 0
    got = oracle.decode_attn(q, K, V, np.array([n], np.int32), dtype, lib=lib)
    for h in range(H):
        want = widen(V[0, h, :n], dtype).mean(axis=0)
        assert np.abs(got[0, h] - want).max() < 1e-12, "a zero query must give the mean of V"


def pin_dominant_score(lib, dtype="fp32"):
    B, H, H_kv, d, ctx, n, star = 1, 1, 1, 4, 6, 6, 3
    q = np.zeros((B, H, d), np.float32)
    q[0, 0, 0] = 20.0
    K = np.zeros((B, H_kv, ctx, d), np.float32)
    K[0, 0, :, 0] = 0.1
    K[0, 0, star, 0] = 30.0                     # score 300 vs 1 for the rest
    V = synth.to_bits(synth.normal((B, H_kv, ctx, d), "fp32", 19))
    got = oracle.decode_attn(q, K, V, np.array([n], np.int32), "fp32", lib=lib)
    assert np.abs(got[0, 0] - V[0, 0, star]).max() < 1e-12, "dominant score must select its V row"


def pin_cached_equals_uncached(lib, dtype="bf16", T=24, H=6, H_kv=3, d=16):
    Q = synth.to_bits(synth.normal((T, H, d), dtype, 23))
    Kt = synth.to_bits(synth.normal((T, H_kv, d), dtype, 29))
    Vt = synth.to_bits(synth.normal((T, H_kv, d), dtype, 31))
    full = oracle.causal_attention(widen(Q, dtype), widen(Kt, dtype), widen(Vt, dtype))
    # cache layout [B=1, H_kv, ctx=T, d]; step t has rows 0..t live
    K = np.ascontiguousarray(np.transpose(Kt, (1, 0, 2))[None])
    V = np.ascontiguousarray(np.transpose(Vt, (1, 0, 2))[None])
    for t in range(T):
        got = oracle.decode_attn(Q[t][None], K, V, np.array([t + 1], np.int32), dtype, lib=lib)
        err = np.abs(got[0] - full[t]).max()
        assert err < 1e-12, f"step {t}: cached decode differs from causal row ({err})"


def pin_gqa_equals_repeated_mha(lib, dtype="bf16", B=2, H=8, H_kv=2, d=16, ctx=20):
    q, K, V = _inputs(dtype, B, H, H_kv, d, ctx, 37)
    valid = np.array([ctx, 5], np.int32)
    g = H // H_kv
    got = oracle.decode_attn(q, K, V, valid, dtype, lib=lib)
    Kr = np.ascontiguousarray(np.repeat(K, g, axis=1))
    Vr = np.ascontiguousarray(np.repeat(V, g, axis=1))
    mha = oracle.decode_attn(q, Kr, Vr, valid, dtype, lib=lib)
    assert np.array_equal(got, mha), "GQA must equal MHA over repeated KV heads"


def brute_force(q, K, V, valid, dtype):
    """Python floats and math.exp; softmax as exp(s) / sum(exp(s))."""
    B, H, d = q.shape
    H_kv = K.shape[1]
    g = H // H_kv
    qf, Kf, Vf = widen(q, dtype), widen(K, dtype), widen(V, dtype)
    out = np.zeros((B, H, d))
    for b in range(B):
        for h in range(H):
            kv = h // g
            e = []
            for j in range(int(valid[b])):
                s = sum(float(qf[b, h, i]) * float(Kf[b, kv, j, i]) for i in range(d))
                e.append(math.exp(s / math.sqrt(d)))
            z = sum(e)
            for i in range(d):
                out[b, h, i] = sum(e[j] * float(Vf[b, kv, j, i]) for j in range(len(e))) / z
    return out


def pin_brute_force(lib, dtype="fp16", B=2, H=4, H_kv=2, d=8, ctx=16):
    q, K, V = _inputs(dtype, B, H, H_kv, d, ctx, 41)
    valid = np.array([16, 3], np.int32)
    got = oracle.decode_attn(q, K, V, valid, dtype, lib=lib)
    ref = brute_force(q, K, V, valid, dtype)
    err = np.abs(got - ref).max()
    assert err < 1e-12, f"oracle vs brute force: {err}"


def pin_widening(lib):
    for dtype, tdt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
        ref = torch.from_numpy(bits.view(np.int16)).view(tdt).to(torch.float64).numpy()
        got = np.array([lib.kvo_widen(bits.ctypes.data, i, oracle.DTYPE_CODES[dtype])
                        for i in range(0, 1 << 16, 7)])
        sub = ref[::7]
        nan = np.isnan(sub)
        assert np.array_equal(np.isnan(got), nan), f"{dtype} NaN set differs"
        assert np.array_equal(got[~nan], sub[~nan]), f"{dtype} widening differs from torch"


ALL_PINS = [pin_library_sdpa, pin_single_row, pin_equal_keys_mean, pin_zero_query_mean,
            pin_dominant_score, pin_cached_equals_uncached, pin_gqa_equals_repeated_mha,
            pin_brute_force, pin_widening]
