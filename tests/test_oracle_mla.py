"""Pins of the MLA decode oracle (oracle.mla_decode_attn).

"10.3 -- KV cache implementation details", section 4.3: one cached latent
per token, keys and values rebuilt per head by up-projections.  The oracle is
pinned by what the mathematics fixes independently of its own code path:
* identity up-projections (d_c = d_h) turn it into multi-query attention
  over the latents, which the separately pinned decode oracle computes;
* the absorbed evaluation order (the projection folded into the query, the
  attention over the latents, the value projection applied last) agrees to
  rounding;
* one live row gives W_UV[h] @ c_0 whatever the query; identical live
  latents give that too; a zero query gives W_UV[h] @ mean(c);
* a pure-Python brute force (explicit rebuilt rows, math.exp, no max shift)
  on tiny shapes;
* planted mistakes (value projection used for the keys, heads' projections
  shifted, the newest latent dropped, the scale taken from d_c) each fail at
  least one of these.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import mla
from oracle.causal import widen


def _bf16(x):
    """float -> bf16 bits (round to nearest even), numpy only."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _inputs(B, H, d_h, d_c, ctx, seed, dtype="fp32"):
    g = np.random.default_rng(seed)
    q = g.standard_normal((B, H, d_h))
    C = g.standard_normal((B, ctx, d_c))
    wk = g.standard_normal((H, d_h, d_c)) / np.sqrt(d_c)
    wv = g.standard_normal((H, d_h, d_c)) / np.sqrt(d_c)
    if dtype == "bf16":
        return _bf16(q), _bf16(C), _bf16(wk), _bf16(wv)
    return q.astype(np.float32), C.astype(np.float32), wk.astype(np.float32), wv.astype(np.float32)


def _absorbed(q, C, wk, wv, valid, dtype):
    """The absorbed order, in numpy: q~ = W_UK^T q, attention of q~ over the
    latents scaled by 1/sqrt(d_h), then W_UV applied to the attended latent."""
    q, C, wk, wv = (widen(a, dtype) for a in (q, C, wk, wv))
    B, H, d_h = q.shape
    out = np.empty((B, H, d_h))
    for b in range(B):
        c = C[b, :valid[b]]
        for h in range(H):
            qt = wk[h].T @ q[b, h]
            s = c @ qt / np.sqrt(d_h)
            w = np.exp(s - s.max())
            o_lat = (w / w.sum()) @ c
            out[b, h] = wv[h] @ o_lat
    return out


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_identity_projections_give_mqa_over_the_latents(dtype):
    B, H, d, ctx = 3, 4, 16, 40
    q, C, _, _ = _inputs(B, H, d, d, ctx, seed=1, dtype=dtype)
    eye = np.broadcast_to(np.eye(d, dtype=np.float32), (H, d, d))
    eye = _bf16(eye) if dtype == "bf16" else np.ascontiguousarray(eye)
    valid = np.array([40, 1, 17])
    got = oracle.mla_decode_attn(q, C, eye, eye, valid, dtype)
    ref = oracle.decode_attn(q, np.ascontiguousarray(C[:, None]), np.ascontiguousarray(C[:, None]), valid, dtype)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("shape", [(2, 4, 8, 32, 50), (1, 16, 16, 64, 130), (3, 2, 32, 24, 9)])
def test_absorbed_order_agrees(shape):
    B, H, d_h, d_c, ctx = shape
    q, C, wk, wv = _inputs(B, H, d_h, d_c, ctx, seed=sum(shape))
    valid = np.linspace(1, ctx, B).astype(np.int32)
    got = oracle.mla_decode_attn(q, C, wk, wv, valid, "fp32")
    np.testing.assert_allclose(got, _absorbed(q, C, wk, wv, valid, "fp32"), rtol=0, atol=1e-12)


def test_closed_forms():
    B, H, d_h, d_c, ctx = 2, 4, 8, 12, 30
    q, C, wk, wv = _inputs(B, H, d_h, d_c, ctx, seed=7)
    W = widen(wv, "fp32")
    c = widen(C, "fp32")
    # one live row: W_UV[h] c_0 whatever the query
    got = oracle.mla_decode_attn(q, C, wk, wv, np.array([1, 1]), "fp32")
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(got[b, h], W[h] @ c[b, 0], rtol=0, atol=1e-14)
    # identical live latents: the same
    Ceq = np.repeat(C[:, :1], ctx, axis=1)
    got = oracle.mla_decode_attn(q, Ceq, wk, wv, np.array([30, 9]), "fp32")
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(got[b, h], W[h] @ c[b, 0], rtol=0, atol=1e-13)
    # zero query: W_UV[h] applied to the mean live latent
    valid = np.array([30, 9])
    got = oracle.mla_decode_attn(np.zeros_like(q), C, wk, wv, valid, "fp32")
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(got[b, h], W[h] @ c[b, :valid[b]].mean(axis=0), rtol=0, atol=1e-13)


def _brute(q, C, wk, wv, valid):
    """Pure Python: rebuild each key and value row element by element, then
    the softmax weights as exp(s) / sum exp(s) without a max shift."""
    B, H, d_h = len(q), len(q[0]), len(q[0][0])
    d_c = len(C[0][0])
    out = []
    for b in range(B):
        ob = []
        for h in range(H):
            ks = [[sum(wk[h][i][j] * C[b][t][j] for j in range(d_c)) for i in range(d_h)] for t in range(valid[b])]
            vs = [[sum(wv[h][i][j] * C[b][t][j] for j in range(d_c)) for i in range(d_h)] for t in range(valid[b])]
            e = [math.exp(sum(q[b][h][i] * k[i] for i in range(d_h)) / math.sqrt(d_h)) for k in ks]
            z = sum(e)
            ob.append([sum(e[t] * vs[t][i] for t in range(valid[b])) / z for i in range(d_h)])
        out.append(ob)
    return np.array(out)


def test_brute_force_tiny():
    B, H, d_h, d_c, ctx = 2, 3, 4, 5, 7
    q, C, wk, wv = _inputs(B, H, d_h, d_c, ctx, seed=11)
    valid = [7, 3]
    ref = _brute(*(widen(a, "fp32").tolist() for a in (q, C, wk, wv)), valid)
    got = oracle.mla_decode_attn(q, C, wk, wv, np.array(valid), "fp32")
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


# ---- planted mistakes: each must break at least one pin above
def _mutant(kind):
    def f(q, C, W_UK, W_UV, valid_len, dtype):
        if kind == "v_for_k":
            W_UK = W_UV
        elif kind == "heads_shifted":
            W_UK, W_UV = np.roll(W_UK, 1, axis=0), np.roll(W_UV, 1, axis=0)
        elif kind == "newest_dropped":
            valid_len = np.maximum(np.asarray(valid_len) - 1, 1)
        K, V = mla.rebuild_kv(np.asarray(C), W_UK, W_UV, dtype)
        qd = widen(q, dtype)
        if kind == "scale_from_d_c":
            qd = qd * np.sqrt(qd.shape[-1] / np.asarray(C).shape[-1])
        return oracle.decode_attn(qd, K, V, np.asarray(valid_len, dtype=np.int32), "fp64")
    return f


@pytest.mark.parametrize("kind", ["v_for_k", "heads_shifted", "newest_dropped", "scale_from_d_c"])
def test_planted_mistakes_are_caught(kind):
    bad = _mutant(kind)
    B, H, d_h, d_c, ctx = 2, 4, 8, 32, 50
    q, C, wk, wv = _inputs(B, H, d_h, d_c, ctx, seed=21)
    valid = np.array([50, 13])
    caught = not np.allclose(bad(q, C, wk, wv, valid, "fp32"), _absorbed(q, C, wk, wv, valid, "fp32"), atol=1e-9)
    tq, tC, twk, twv = _inputs(1, 2, 3, 4, 6, seed=22)
    caught |= not np.allclose(bad(tq, tC, twk, twv, np.array([6]), "fp32"),
                              _brute(*(widen(a, "fp32").tolist() for a in (tq, tC, twk, twv)), [6]), atol=1e-9)
    assert caught, kind
    # and the unaltered oracle passes the same checks
    assert np.allclose(oracle.mla_decode_attn(q, C, wk, wv, valid, "fp32"), _absorbed(q, C, wk, wv, valid, "fp32"),
                       atol=1e-9)
