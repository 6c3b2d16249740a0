"""kvc_decode_step -- the whole decode step of one layer in one call.

"10.3 -- KV cache implementation details", section 5 (the decode loop): the
step appends k_t, v_t to the layer's cache, then the single query row attends
over the entire cache.  kvc_decode_step does both in one launch that takes
the new rows from k_new / v_new directly (on the tensor-core kernels and on
the CUDA-core kernel alike).  Checked here: the cache bytes after the step equal those of
a list-append cache (bit-exact, padded rows still poisoned), the output
matches the fp64 oracle within the decode tolerances, and the fused launch
agrees with append + decode_attn wherever the new row falls in a tile or a
split.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import ListAppendCache
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


def _dense_bits(lc, layer, which, ctx, dtype):
    u8 = lc.dense(layer, which, ctx)
    return u8.view(np.float32 if dtype == "fp32" else np.uint16)


def _mirror_prefix(hn, lc, layer, lengths):
    """Copy rows [0, lengths[b]) that fill_prefix wrote into the list cache."""
    w = hn.w
    for b in range(w.batch):
        n = int(lengths[b])
        if n == 0:
            continue
        kb = _gpu.bits(hn.K[layer, b, :, :n]).view(np.uint8).reshape(w.n_kv_heads, n, w.row_bytes)
        vb = _gpu.bits(hn.V[layer, b, :, :n]).view(np.uint8).reshape(w.n_kv_heads, n, w.row_bytes)
        for kv in range(w.n_kv_heads):
            for t in range(n):
                lc.k[layer][b][kv].append(kb[kv, t].tobytes())
                lc.v[layer][b][kv].append(vb[kv, t].tobytes())


def _check_cache(hn, lc, layer, lengths, dtype):
    """Live rows equal the list-append cache bit for bit; the row after the
    live ones still holds the poison pattern."""
    w = hn.w
    poison = synth.POISON_BITS[dtype]
    it = np.uint32 if dtype == "fp32" else np.uint16  # compare bit patterns
    kh = _gpu.bits(hn.K[layer]).view(it)
    vh = _gpu.bits(hn.V[layer]).view(it)
    ctx = int(max(lengths))
    kd = _dense_bits(lc, layer, "k", ctx, dtype).view(it)
    vd = _dense_bits(lc, layer, "v", ctx, dtype).view(it)
    for b in range(w.batch):
        n = int(lengths[b])
        assert np.array_equal(kh[b, :, :n], kd[b, :, :n]), f"K rows of sequence {b}"
        assert np.array_equal(vh[b, :, :n], vd[b, :, :n]), f"V rows of sequence {b}"
        if n < w.max_context:
            assert (kh[b, :, n] == poison).all() and (vh[b, :, n] == poison).all()


# Sequences of steps on every kernel (all of them fuse the step's append).
SEQ = [
    # name, dtype, d_h, H, H_kv, B, max_ctx, prefilled rows per sequence
    ("bf16_g4_d128", "bf16", 128, 16, 4, 5, 700, [0, 31, 32, 250, 690]),
    ("fp16_g6_d64", "fp16", 64, 12, 2, 3, 300, [7, 64, 200]),
    ("bf16_g8_d128", "bf16", 128, 8, 1, 2, 520, [1, 480]),
    ("bf16_g32_d128_mqa", "bf16", 128, 32, 1, 3, 600, [0, 33, 590]),
    ("fp16_g16_d64", "fp16", 64, 32, 2, 2, 400, [64, 391]),
    ("fp16_g16_d128_tc", "fp16", 128, 32, 2, 3, 400, [0, 127, 383]),
    ("fp32_g6_d128_cuda_core", "fp32", 128, 12, 2, 3, 300, [0, 40, 290]),
    ("bf16_g1_d128_cuda_core", "bf16", 128, 4, 4, 2, 300, [5, 100]),
    ("bf16_g4_d32_cuda_core", "bf16", 32, 16, 4, 3, 200, [0, 63, 190]),
]


@pytest.mark.parametrize("case", SEQ, ids=[c[0] for c in SEQ])
def test_step_sequence_matches_oracle(case):
    name, dtype, D, H, H_kv, B, T, pre = case
    steps, L = 6, 2
    w = synth.Workload(name, L, B, H, H_kv, D, T, dtype, steps=steps, seed=900 + len(name))
    hn = _gpu.Harness(w)
    lc = ListAppendCache(L, B, H_kv, w.row_bytes)
    for layer in range(L):
        _gpu.fill_prefix(hn, layer, pre, "pre")
        _mirror_prefix(hn, lc, layer, pre)
    lengths = np.array(pre, dtype=np.int64)
    for step in range(steps):
        ci = lengths.copy()
        lengths = lengths + 1
        valid = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        for layer in range(L):
            k, v = _gpu.new_rows(w, 1, "step", step, layer)
            q = _gpu.query(w, "step", step, layer)
            st, out = hn.step(layer, q, k, v, valid, hint=int(lengths.max()))
            assert st == 0
            lc.append(layer, _gpu.bits(k), _gpu.bits(v), ci, 1)
            ctx = int(lengths.max())
            ref = oracle.decode_attn(_gpu.bits(q), _dense_bits(lc, layer, "k", ctx, dtype),
                                     _dense_bits(lc, layer, "v", ctx, dtype), lengths, dtype)
            _gpu.compare(out, ref, dtype, f"{name} step {step} layer {layer}")
    assert hn.error() == 0
    for layer in range(L):
        _check_cache(hn, lc, layer, lengths, dtype)
    assert hn.canaries_intact()


# New rows at every interesting offset: first row, ends and starts of 8-row
# groups and of 32-row tiles, near split boundaries, the last row of the buffer.
EDGE_LENGTHS = [1, 2, 8, 9, 31, 32, 33, 40, 64, 65, 511, 700]


@pytest.mark.parametrize("splits", [0, 1, 3, 13, 152])
@pytest.mark.parametrize("dtype,D,H,H_kv", [("bf16", 128, 16, 4), ("fp16", 64, 6, 2), ("bf16", 128, 32, 1),
                                           ("fp16", 128, 32, 2),
                                           # the CUDA-core kernel: fp32, one head per KV head, d_h 32 / 256
                                           ("fp32", 128, 8, 2), ("bf16", 128, 8, 8), ("fp16", 32, 4, 4),
                                           ("bf16", 256, 4, 2)])
def test_fused_step_equals_append_then_decode(splits, dtype, D, H, H_kv):
    B, T = len(EDGE_LENGTHS), 700
    w = synth.Workload(f"edge_{dtype}", 1, B, H, H_kv, D, T, dtype, steps=1, seed=931)
    fused, twice = _gpu.Harness(w), _gpu.Harness(w)
    lengths = np.array(EDGE_LENGTHS, dtype=np.int64)
    for hn in (fused, twice):
        _gpu.fill_prefix(hn, 0, lengths - 1, "edge")
        if splits:
            assert hn.kvc.kvc_set_num_splits(hn.h, splits) == 0
    k, v = _gpu.new_rows(w, 1, "edge")
    q = _gpu.query(w, "edge")
    valid = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    st, out_fused = fused.step(0, q, k, v, valid, hint=T)
    assert st == 0
    assert twice.append(0, k, v, (valid - 1), 1) == 0
    st, out_twice = twice.decode(0, q, valid, hint=T)
    assert st == 0
    assert fused.error() == 0 and twice.error() == 0
    # identical cache bytes, padded rows included
    assert torch.equal(fused.K.view(torch.uint8), twice.K.view(torch.uint8))
    assert torch.equal(fused.V.view(torch.uint8), twice.V.view(torch.uint8))
    Kh, Vh = _gpu.bits(twice.K[0]), _gpu.bits(twice.V[0])
    ref = oracle.decode_attn(_gpu.bits(q), Kh, Vh, lengths, dtype)
    _gpu.compare(out_fused, ref, dtype, "fused step")
    _gpu.compare(out_twice, ref, dtype, "append + decode")
    assert fused.canaries_intact() and twice.canaries_intact()


@pytest.mark.parametrize("dtype,H,H_kv", [("bf16", 8, 2), ("fp32", 8, 2)])
def test_step_bad_valid_len_skips_append_and_output(dtype, H, H_kv):
    w = synth.Workload("step_bad", 1, 3, H, H_kv, 128, 100, dtype, steps=1, seed=941)
    hn = _gpu.Harness(w)
    pre = [49, 10, 99]
    _gpu.fill_prefix(hn, 0, pre, "bad")
    before = hn.K.clone(), hn.V.clone()
    k, v = _gpu.new_rows(w, 1, "bad")
    q = _gpu.query(w, "bad")
    for bad in (0, 101, -3):
        vl = torch.tensor([50, bad, 100], dtype=torch.int32, device="cuda")
        out = torch.full((w.batch, w.n_heads, w.d_head), 7.0, device="cuda").to(synth.DTYPES[dtype])
        st, out = hn.step(0, q, k, v, vl, hint=100, out=out)
        assert st == 0
        assert hn.error() == hn.kvc.KVC_ERR_DEVICE_INDEX
        assert (out[1].float() == 7.0).all(), "a skipped sequence's output must stay unwritten"
        assert torch.equal(hn.K[0, 1].view(torch.uint8), before[0][0, 1].view(torch.uint8))
        assert torch.equal(hn.V[0, 1].view(torch.uint8), before[1][0, 1].view(torch.uint8))
    good = [0, 2]
    Kh, Vh = _gpu.bits(hn.K[0]).copy(), _gpu.bits(hn.V[0]).copy()
    ref = oracle.decode_attn(_gpu.bits(q)[good], Kh[good], Vh[good], np.array([50, 100]), dtype)
    _gpu.compare(out[good], ref, dtype, "the valid sequences")
    assert hn.canaries_intact()


def test_step_host_errors():
    w = synth.Workload("step_err", 1, 2, 8, 2, 128, 64, "bf16", steps=1, seed=951)
    hn = _gpu.Harness(w)
    kvc = hn.kvc
    k, v = _gpu.new_rows(w, 1, "err")
    q = _gpu.query(w, "err")
    vl = torch.ones(2, dtype=torch.int32, device="cuda")
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    assert kvc.kvc_decode_step(hn.h, 0, q, 0, v, vl, 1, out, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_decode_step(hn.h, 0, q, k, 0, vl, 1, out, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_decode_step(hn.h, 1, q, k, v, vl, 1, out, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_decode_step(hn.h, 0, q, k, v, vl, 65, out, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_decode_step(hn.h, 0, q, k.data_ptr() + 2, v, vl, 1, out, None) == kvc.KVC_ERR_ALIGNMENT
    assert kvc.kvc_decode_step(None, 0, q, k, v, vl, 1, out, None) == kvc.KVC_ERR_INVALID
    assert hn.error() == 0


@pytest.mark.parametrize("layers", [(0, 31)])
def test_full_size_fused_step_llama3(layers):
    """The bench's configuration: the Llama-3-shaped cache (32 layers, B=16,
    ragged U{1024..8192}) stepped through kvc_decode_step, one fused launch
    per layer; sampled layers checked against the oracle and the new rows
    checked in place."""
    w = synth.WORKLOADS["llama3_8b"]
    hn = _gpu.Harness(w)
    lengths = synth.live_lengths(w)
    pre = (lengths - 1).tolist()
    maxlen = int(lengths.max())
    host = {}
    for layer in layers:
        _gpu.fill_prefix(hn, layer, pre)
        host[layer] = (_gpu.bits(hn.K[layer, :, :, :maxlen]).copy(), _gpu.bits(hn.V[layer, :, :, :maxlen]).copy())
    valid = lengths.cuda()
    for layer in layers:
        k, v = _gpu.new_rows(w, 1, "full-step", layer)
        q = _gpu.query(w, "full-step", layer)
        st, out = hn.step(layer, q, k, v, valid, hint=maxlen)
        assert st == 0
        Kh, Vh = host[layer]
        kb, vb = _gpu.bits(k), _gpu.bits(v)
        for b in range(w.batch):
            Kh[b, :, pre[b]] = kb[b, :, 0]
            Vh[b, :, pre[b]] = vb[b, :, 0]
            assert np.array_equal(_gpu.bits(hn.K[layer, b, :, pre[b]]), kb[b, :, 0]), "new K row in place"
            assert np.array_equal(_gpu.bits(hn.V[layer, b, :, pre[b]]), vb[b, :, 0]), "new V row in place"
        ref = oracle.decode_attn(_gpu.bits(q), Kh, Vh, lengths.numpy(), w.dtype)
        _gpu.compare(out, ref, w.dtype, f"fused step, layer {layer}")
    assert hn.error() == 0
    assert hn.canaries_intact()
