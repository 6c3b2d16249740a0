"""Decode attention on the GPU against the fp64 oracle.

"10.3 -- KV cache implementation details", section 5: one query row per
head attends over the whole cache, softmax(q K^T / sqrt(d_head)) V; GQA
shares each KV head across the group (section 4.2).  Tolerances: bf16 and
fp16 outputs within 2e-2 absolute, fp32 within 1e-5 of each row's largest
magnitude.  Every cache row past the live length holds a NaN pattern, so a
read of a padded row would surface as a non-finite output.
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


# --------------------------------------------------------------------------
# The two small workloads, every step, through append + decode.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny_mha", "small_gqa"])
def test_decode_sequence_matches_oracle(name):
    w = synth.WORKLOADS[name]
    hn = _gpu.Harness(w)
    lc = ListAppendCache(w.n_layers, w.batch, w.n_kv_heads, w.row_bytes)
    first = w.first_append or w.prefill
    for layer in range(w.n_layers):
        k, v = _gpu.new_rows(w, first, "first", layer)
        ci = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
        assert hn.append(layer, k, v, ci, first) == 0
        lc.append(layer, _gpu.bits(k), _gpu.bits(v), [0] * w.batch, first)
    worst = 0.0
    for step in range(w.steps):
        pos = first + step
        ci = torch.full((w.batch,), pos, dtype=torch.int32, device="cuda")
        valid = torch.full((w.batch,), pos + 1, dtype=torch.int32, device="cuda")
        for layer in range(w.n_layers):
            k, v = _gpu.new_rows(w, 1, step, layer)
            q = _gpu.query(w, step, layer)
            assert hn.append(layer, k, v, ci, 1) == 0
            st, out = hn.decode(layer, q, valid, hint=pos + 1)
            assert st == 0
            lc.append(layer, _gpu.bits(k), _gpu.bits(v), [pos] * w.batch, 1)
            ctx = pos + 1
            ref = oracle.decode_attn(_gpu.bits(q), _dense_bits(lc, layer, "k", ctx, w.dtype),
                                     _dense_bits(lc, layer, "v", ctx, w.dtype),
                                     [ctx] * w.batch, w.dtype)
            worst = max(worst, _gpu.compare(out, ref, w.dtype, f"{name} step {step} layer {layer}"))
    assert hn.error() == 0
    assert hn.canaries_intact()


def test_tiny_cached_equals_uncached_causal():
    """Every decode step of the tiny workload equals the matching row of full
    causal attention recomputed over all tokens ("KV-Cache Mechanics",
    Disabling the Cache)."""
    w = synth.WORKLOADS["tiny_mha"]
    T = 80
    hn = _gpu.Harness(w)
    q_all = synth.normal((T, w.n_heads, w.d_head), w.dtype, synth.sub_seed(w.seed, "cq"), device="cuda")
    k_all = synth.normal((T, w.n_kv_heads, w.d_head), w.dtype, synth.sub_seed(w.seed, "ck"), device="cuda")
    v_all = synth.normal((T, w.n_kv_heads, w.d_head), w.dtype, synth.sub_seed(w.seed, "cv"), device="cuda")
    full = oracle.causal_attention(oracle.widen(_gpu.bits(q_all), w.dtype),
                                   oracle.widen(_gpu.bits(k_all), w.dtype),
                                   oracle.widen(_gpu.bits(v_all), w.dtype))
    for t in range(T):
        k = k_all[t].reshape(1, w.n_kv_heads, 1, w.d_head).contiguous()
        v = v_all[t].reshape(1, w.n_kv_heads, 1, w.d_head).contiguous()
        assert hn.append(0, k, v, torch.tensor([t], dtype=torch.int32, device="cuda"), 1) == 0
        st, out = hn.decode(0, q_all[t][None].contiguous(), torch.tensor([t + 1], dtype=torch.int32,
                                                                       device="cuda"), hint=t + 1)
        assert st == 0
        _gpu.compare(out[0], full[t], w.dtype, f"causal row {t}")
    assert hn.error() == 0


# --------------------------------------------------------------------------
# Full-size workloads: one decode step (append at valid - 1, then attend).
# --------------------------------------------------------------------------
def _one_step(w, check_layers):
    hn = _gpu.Harness(w)
    lengths = synth.live_lengths(w)
    pre = (lengths - 1).tolist()
    maxlen = int(lengths.max())
    host_prefix = {}
    for layer in range(w.n_layers):
        _gpu.fill_prefix(hn, layer, pre)
        if layer in check_layers:
            host_prefix[layer] = (_gpu.bits(hn.K[layer, :, :, :maxlen]).copy(),
                                  _gpu.bits(hn.V[layer, :, :, :maxlen]).copy())
    torch.cuda.synchronize()
    ci = (lengths - 1).cuda()
    valid = lengths.cuda()
    kept = {}
    for layer in range(w.n_layers):
        k, v = _gpu.new_rows(w, 1, "step", layer)
        q = _gpu.query(w, "step", layer)
        assert hn.append(layer, k, v, ci, 1) == 0
        st, out = hn.decode(layer, q, valid, hint=maxlen)
        assert st == 0
        kept[layer] = (k, v, q, out)
    assert hn.error() == 0
    # append: the new rows are in place in every layer, neighbours untouched
    poison = synth.POISON_BITS[w.dtype]
    for layer in range(w.n_layers):
        k, v, _, _ = kept[layer]
        for b in range(w.batch):
            p = pre[b]
            assert torch.equal(hn.K[layer, b, :, p].contiguous().view(torch.uint8),
                               k[b, :, 0].contiguous().view(torch.uint8))
            assert torch.equal(hn.V[layer, b, :, p].contiguous().view(torch.uint8),
                               v[b, :, 0].contiguous().view(torch.uint8))
            if p + 1 < w.max_context:
                row = _gpu.bits(hn.K[layer, b, :, p + 1])
                assert (row.view(np.uint32 if w.dtype == "fp32" else np.uint16) == poison).all()
    # attention: oracle over prefix + appended row
    for layer in check_layers:
        k, v, q, out = kept[layer]
        Kh, Vh = host_prefix[layer]
        kb, vb = _gpu.bits(k), _gpu.bits(v)
        for b in range(w.batch):
            Kh[b, :, pre[b]] = kb[b, :, 0]
            Vh[b, :, pre[b]] = vb[b, :, 0]
        ref = oracle.decode_attn(_gpu.bits(q), Kh, Vh, lengths.numpy(), w.dtype)
        _gpu.compare(out, ref, w.dtype, f"{w.name} layer {layer}")
    assert hn.canaries_intact()


@pytest.mark.parametrize("name,layers", [
    ("llama3_8b", (0, 1, 31)),
    ("qwen2_5_1_5b_fp32", (0, 27)),
    ("qwen2_5_1_5b_bf16", (0, 27)),
    ("llama2_70b_b1", (0,)),
    ("llama2_70b_b4", (0,)),
])
def test_full_size_one_step(name, layers):
    _one_step(synth.WORKLOADS[name], layers)


def test_full_size_mqa_one_step():
    """The benchmarked multi-query shape (32 query heads on one KV head,
    B=128, ragged U{1024..8192}), two of its layers: every sequence's append
    and the whole layer's attention against the oracle."""
    _one_step(synth.WORKLOADS["mqa_32h"].with_(n_layers=2), (1,))


# --------------------------------------------------------------------------
# Shapes spanning several tiles, ragged tails, every element type and
# several head groups / widths, with the automatic and forced split counts.
# --------------------------------------------------------------------------
CASES = [
    # dtype, d, H, H_kv, B, max_ctx, seed
    ("bf16", 128, 32, 8, 5, 3000, 1),
    ("bf16", 128, 8, 8, 2, 5000, 2),
    ("fp32", 128, 12, 2, 3, 2048, 3),
    ("fp16", 64, 16, 4, 3, 1500, 4),
    ("bf16", 32, 8, 2, 4, 700, 5),
    ("bf16", 256, 8, 1, 2, 1000, 6),
    ("fp32", 256, 6, 2, 2, 600, 7),
    ("bf16", 128, 7, 1, 3, 900, 8),
    ("fp16", 128, 5, 5, 2, 400, 9),
    ("fp32", 32, 3, 1, 3, 333, 10),
    ("bf16", 64, 12, 4, 6, 1200, 11),
    ("fp16", 256, 16, 2, 2, 257, 12),
    # head groups of 16, 32 and 64 ("10.3", section 4.1: multi-query
    # attention, one KV head shared by every query head)
    ("bf16", 128, 32, 1, 4, 2500, 13),
    ("bf16", 128, 32, 2, 3, 1800, 14),
    ("fp16", 64, 16, 1, 5, 1200, 15),
    ("bf16", 128, 64, 1, 2, 1300, 16),
    ("fp16", 128, 64, 2, 2, 900, 17),
    # 16 and 32 heads at d_h 128 run the tcgen05 kernel: fp16, and 16 heads
    ("fp16", 128, 32, 1, 3, 2100, 18),
    ("fp16", 128, 16, 2, 4, 1500, 19),
    ("bf16", 128, 16, 1, 5, 700, 20),
]


def _ragged_case(dtype, d, H, H_kv, B, max_ctx, seed, splits_list):
    w = synth.Workload(f"case{seed}", 1, B, H, H_kv, d, max_ctx, dtype, steps=1,
                       ragged=(1, max_ctx), seed=100 + seed)
    hn = _gpu.Harness(w)
    lengths = synth.live_lengths(w)
    lengths[0] = max_ctx                       # one sequence at full capacity
    if B > 2:
        lengths[1] = 1                         # and one with a single live row
    _gpu.fill_prefix(hn, 0, (lengths - 1).tolist())
    torch.cuda.synchronize()
    k, v = _gpu.new_rows(w, 1, "x")
    q = _gpu.query(w, "x")
    maxlen = int(lengths.max())
    Kh = _gpu.bits(hn.K[0, :, :, :maxlen]).copy()     # the prefix, before any library kernel
    Vh = _gpu.bits(hn.V[0, :, :, :maxlen]).copy()
    kb, vb = _gpu.bits(k), _gpu.bits(v)
    for b in range(B):
        Kh[b, :, int(lengths[b]) - 1] = kb[b, :, 0]
        Vh[b, :, int(lengths[b]) - 1] = vb[b, :, 0]
    assert hn.append(0, k, v, (lengths - 1).cuda(), 1) == 0
    ref = oracle.decode_attn(_gpu.bits(q), Kh, Vh, lengths.numpy(), dtype)
    outs = []
    for splits in splits_list:
        assert hn.kvc.kvc_set_num_splits(hn.h, splits) == 0
        st, out = hn.decode(0, q, lengths.cuda(), hint=maxlen)
        assert st == 0
        _gpu.compare(out, ref, dtype, f"{w.name} splits={splits}")
        outs.append(out.float())
    assert hn.error() == 0
    assert hn.canaries_intact()
    return outs


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_d{c[1]}_H{c[2]}_Hkv{c[3]}_B{c[4]}" for c in CASES])
def test_ragged_shapes_against_oracle(case):
    _ragged_case(*case, splits_list=[0, 1, 3, 152, 1024])


def test_split_count_changes_only_rounding():
    """One split and many splits agree to fp32 rounding (fp32 cache)."""
    outs = _ragged_case("fp32", 128, 8, 2, 3, 4000, 21, splits_list=[1, 2, 17, 300])
    for o in outs[1:]:
        rel = ((o - outs[0]).abs().max() / outs[0].abs().max()).item()
        assert rel < 2e-6, rel


def test_single_live_row_returns_v_exactly():
    """valid = 1: the softmax weight is exactly 1, so out is the V row."""
    w = synth.Workload("one_row", 1, 3, 8, 2, 128, 64, "bf16", steps=1, seed=31)
    hn = _gpu.Harness(w)
    k, v = _gpu.new_rows(w, 1, "one")
    q = _gpu.query(w, "one")
    ci = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
    assert hn.append(0, k, v, ci, 1) == 0
    st, out = hn.decode(0, q, torch.ones(w.batch, dtype=torch.int32, device="cuda"), hint=1)
    assert st == 0
    want = v[:, :, 0].repeat_interleave(w.group, dim=1)
    assert torch.equal(out.view(torch.int16), want.contiguous().view(torch.int16))


def test_mqa_equals_mha_on_repeated_heads():
    """Multi-query attention (one KV head for all 32 query heads) equals MHA
    over a cache holding that head repeated 32 times ("10.3", section 4.1)."""
    g = 32
    wq = synth.Workload("mqa", 1, 3, 32, 1, 128, 900, "bf16", steps=1, seed=42)
    wm = wq.with_(n_kv_heads=32)
    hq, hm = _gpu.Harness(wq), _gpu.Harness(wm)
    lengths = torch.tensor([900, 1, 517], dtype=torch.int32)
    _gpu.fill_prefix(hq, 0, lengths.tolist())
    hm.K[0] = hq.K[0].repeat_interleave(g, dim=1)
    hm.V[0] = hq.V[0].repeat_interleave(g, dim=1)
    q = _gpu.query(wq, "m")
    st, oq = hq.decode(0, q, lengths.cuda(), hint=900)
    assert st == 0
    st, om = hm.decode(0, q, lengths.cuda(), hint=900)
    assert st == 0
    assert (oq.float() - om.float()).abs().max().item() <= 2e-2
    ref = oracle.decode_attn(_gpu.bits(q), _gpu.bits(hq.K[0]).copy(), _gpu.bits(hq.V[0]).copy(),
                             lengths.numpy(), "bf16")
    _gpu.compare(oq, ref, "bf16", "mqa")
    assert hq.error() == 0 and hm.error() == 0


def test_gqa_equals_mha_on_repeated_heads():
    """A GQA cache and an MHA cache holding each KV head repeated g times
    give the same output ("KV Cache Optimization...", #1 Fix)."""
    g = 4
    wg = synth.Workload("gqa", 1, 2, 16, 4, 128, 512, "bf16", steps=1, seed=41)
    wm = wg.with_(n_kv_heads=16)
    hg, hm = _gpu.Harness(wg), _gpu.Harness(wm)
    lengths = torch.tensor([512, 300], dtype=torch.int32)
    _gpu.fill_prefix(hg, 0, lengths.tolist())
    hm.K[0] = hg.K[0].repeat_interleave(g, dim=1)
    hm.V[0] = hg.V[0].repeat_interleave(g, dim=1)
    q = _gpu.query(wg, "g")
    st, og = hg.decode(0, q, lengths.cuda(), hint=512)
    assert st == 0
    st, om = hm.decode(0, q, lengths.cuda(), hint=512)
    assert st == 0
    assert (og.float() - om.float()).abs().max().item() <= 2e-2
    Kh = _gpu.bits(hg.K[0]).copy()
    Vh = _gpu.bits(hg.V[0]).copy()
    ref = oracle.decode_attn(_gpu.bits(q), Kh, Vh, lengths.numpy(), "bf16")
    _gpu.compare(og, ref, "bf16", "gqa")
    _gpu.compare(om, ref, "bf16", "mha on repeated heads")


def test_bad_valid_len_is_reported_and_row_skipped():
    w = synth.Workload("bad_len", 1, 3, 4, 2, 64, 100, "fp32", steps=1, seed=51)
    hn = _gpu.Harness(w)
    lengths = [50, 0, 100]
    _gpu.fill_prefix(hn, 0, [50, 0, 100])
    q = _gpu.query(w, "bad")
    out = torch.full((w.batch, w.n_heads, w.d_head), 7.0, device="cuda")
    for bad in (0, 101, -3):
        vl = torch.tensor([50, bad, 100], dtype=torch.int32, device="cuda")
        st, out = hn.decode(0, q, vl, hint=100, out=out)
        assert st == 0
        assert hn.error() == hn.kvc.KVC_ERR_DEVICE_INDEX
        assert (out[1] == 7.0).all(), "a skipped sequence's output must stay unwritten"
    good = [0, 2]
    Kh = _gpu.bits(hn.K[0]).copy()
    Vh = _gpu.bits(hn.V[0]).copy()
    qb = _gpu.bits(q)
    ref = oracle.decode_attn(qb[good], Kh[good], Vh[good], np.array([50, 100]), "fp32")
    _gpu.compare(out[good], ref, "fp32", "the valid sequences")
    assert hn.canaries_intact()


def test_decode_host_errors():
    w = synth.Workload("dec_err", 2, 2, 4, 2, 64, 32, "bf16", steps=1, seed=3)
    hn = _gpu.Harness(w)
    kvc = hn.kvc
    q = _gpu.query(w, "e")
    vl = torch.ones(w.batch, dtype=torch.int32, device="cuda")
    assert hn.decode(2, q, vl)[0] == kvc.KVC_ERR_INVALID
    assert hn.decode(0, q, vl, hint=33)[0] == kvc.KVC_ERR_INVALID
    assert hn.decode(0, q, vl, hint=-1)[0] == kvc.KVC_ERR_INVALID
    raw = torch.empty(q.numel() * 2 + 16, dtype=torch.uint8, device="cuda")
    assert kvc.kvc_decode_attn(hn.h, 0, raw.data_ptr() + 4, vl, 0, q, None) == kvc.KVC_ERR_ALIGNMENT
    assert kvc.kvc_decode_attn(hn.h, 0, q, None, 0, q, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_set_num_splits(hn.h, 1025) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_set_num_splits(hn.h, -1) == kvc.KVC_ERR_INVALID
    assert hn.error() == 0


def test_alloc_errors():
    from static_kv_cache_gb300 import kvc
    cfg = kvc.make_config(1, 1, 8, 2, 128, 64, "bf16")
    need = kvc.kvc_workspace_bytes(cfg)
    k = torch.empty(kvc.kvc_cache_bytes(cfg) // 2 + 64, dtype=torch.uint8, device="cuda")
    v = torch.empty_like(k)
    ws = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
    assert kvc.kvc_alloc(cfg, k, v, ws, need - 1)[0] == kvc.KVC_ERR_WORKSPACE
    assert kvc.kvc_alloc(cfg, k.data_ptr() + 8, v, ws, need)[0] == kvc.KVC_ERR_ALIGNMENT
    bad = kvc.make_config(1, 1, 8, 3, 128, 64, "bf16")
    assert kvc.kvc_alloc(bad, k, v, ws, need)[0] == kvc.KVC_ERR_INVALID
    unsup = kvc.make_config(1, 1, 12, 1, 128, 64, "bf16")    # g = 12: not a whole number of 8-head chunks
    assert kvc.kvc_alloc(unsup, k, v, ws, need)[0] == kvc.KVC_ERR_UNSUPPORTED
    for g, d, dt in ((16, 32, "bf16"), (32, 128, "fp32"), (128, 128, "bf16")):   # no kernel for these
        assert kvc.kvc_check_config(kvc.make_config(1, 1, g, 1, d, 64, dt)) == kvc.KVC_ERR_UNSUPPORTED
    for g, d in ((16, 64), (32, 128), (64, 128)):
        assert kvc.kvc_check_config(kvc.make_config(1, 1, g, 1, d, 64, "bf16")) == kvc.KVC_OK
    st, h = kvc.kvc_alloc(cfg, k, v, ws, need)
    assert st == 0 and h
    kvc.kvc_free(h)
