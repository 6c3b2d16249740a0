"""The int8 cache on the GPU ("10.3 -- KV cache implementation details",
section 4.4: the cache stored as int8, p = 1).

Rows are quantised as they are appended (symmetric, one fp32 scale per row,
codes rint(x * 127 / absmax) in fp32; the reading in oracle/quant.py) and
the attention reads code * scale.  Checked: the codes and scales written by
kvc_append equal the oracle's bit for bit; decode over a cache filled that
way matches the fp64 oracle over the dequantised rows (bf16 output within
2e-2); kvc_decode_step sequences; the quantisation's effect on attention
against the unquantised cache stays small; host errors.  Scale entries past
the live rows hold a NaN pattern, so a read of a padded row would show up as
a non-finite output.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import dequantize_rows, quantize_rows
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FA5A5A5


class Q8Harness:
    """An int8 cache [L, B, H_kv, T, D] with its two scale arrays, all guarded."""

    def __init__(self, L, B, H, H_kv, D, T, seed):
        from static_kv_cache_gb300 import kvc
        self.kvc = kvc
        self.L, self.B, self.H, self.H_kv, self.D, self.T = L, B, H, H_kv, D, T
        self.seed = seed
        self.cfg = kvc.make_config(L, B, H, H_kv, D, T, "int8")
        n = L * B * H_kv * T
        self.kbuf, self.vbuf = _gpu.Guarded(n * D), _gpu.Guarded(n * D)
        self.ksbuf, self.vsbuf = _gpu.Guarded(n * 4), _gpu.Guarded(n * 4)
        assert kvc.kvc_scale_bytes(self.cfg) == n * 4
        self.K = self.kbuf.view(torch.int8, (L, B, H_kv, T, D))
        self.V = self.vbuf.view(torch.int8, (L, B, H_kv, T, D))
        self.KS = self.ksbuf.view(torch.int32, (L, B, H_kv, T))
        self.VS = self.vsbuf.view(torch.int32, (L, B, H_kv, T))
        self.K.fill_(0x55)
        self.V.fill_(-0x55)
        self.KS.fill_(NAN_BITS)
        self.VS.fill_(NAN_BITS)
        self.ws = _gpu.Guarded(kvc.kvc_workspace_bytes(self.cfg))
        st, self.h = kvc.kvc_alloc_scaled(self.cfg, self.kbuf.ptr(), self.vbuf.ptr(), self.ksbuf.ptr(),
                                          self.vsbuf.ptr(), self.ws.ptr(), self.ws.nbytes)
        kvc.check(st, "kvc_alloc_scaled")

    def rows(self, T_new, *tags, scale=1.0):
        shape = (self.B, self.H_kv, T_new, self.D)
        k = synth.normal(shape, "bf16", synth.sub_seed(self.seed, "k8", *tags), device="cuda") * scale
        v = synth.normal(shape, "bf16", synth.sub_seed(self.seed, "v8", *tags), device="cuda") * scale
        return k.to(torch.bfloat16), v.to(torch.bfloat16)

    def query(self, *tags):
        return synth.normal((self.B, self.H, self.D), "bf16", synth.sub_seed(self.seed, "q8", *tags), device="cuda")

    def dequant(self, layer):
        """Host [B, H_kv, T, D] float64 of the stored codes times scales (rows
        past the live ones come out as NaN)."""
        codes = self.K[layer].cpu().numpy(), self.V[layer].cpu().numpy()
        sc = (self.KS[layer].cpu().numpy().view(np.float32), self.VS[layer].cpu().numpy().view(np.float32))
        return dequantize_rows(codes[0], sc[0]), dequantize_rows(codes[1], sc[1])

    def canaries_intact(self):
        return all(b.canaries_intact() for b in (self.kbuf, self.vbuf, self.ksbuf, self.vsbuf, self.ws))

    def close(self):
        self.kvc.kvc_free(self.h)


def _decode_ref(hn, layer, q, lengths):
    Kd, Vd = hn.dequant(layer)
    qd = oracle.widen(_gpu.bits(q), "bf16")
    return oracle.decode_attn(qd, Kd, Vd, np.asarray(lengths), "fp64")


def test_append_quantises_like_the_oracle():
    hn = Q8Harness(2, 3, 8, 2, 128, 64, seed=2100)
    # rows with mixed magnitudes, an all-zero row, and exact half-to-even ties
    k, v = hn.rows(20, "q", scale=1.0)
    k[0, 0, 3] = 0
    k[1, 1, 5] = torch.tensor([0.5, -0.25] + [0.0] * 126, dtype=torch.bfloat16)   # 0.5*254 = 127, -0.25*254 = -63.5
    v[2] *= 1000
    ci = torch.tensor([0, 7, 44], dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_append(hn.h, 1, k, v, ci, 20, None) == 0
    torch.cuda.synchronize()
    kc, ks = quantize_rows(_gpu.bits(k), "bf16")
    vc, vs = quantize_rows(_gpu.bits(v), "bf16")
    assert kc[1, 1, 5, 1] == -64 and kc[1, 1, 5, 0] == 127
    for b, c in enumerate([0, 7, 44]):
        assert np.array_equal(hn.K[1, b, :, c:c + 20].cpu().numpy(), kc[b])
        assert np.array_equal(hn.V[1, b, :, c:c + 20].cpu().numpy(), vc[b])
        assert np.array_equal(hn.KS[1, b, :, c:c + 20].cpu().numpy().view(np.float32), ks[b])
        assert np.array_equal(hn.VS[1, b, :, c:c + 20].cpu().numpy().view(np.float32), vs[b])
        if c > 0:  # the row before the appended ones is untouched
            assert (hn.KS[1, b, :, c - 1].cpu().numpy() == NAN_BITS).all()
    assert (hn.KS[0].cpu().numpy() == NAN_BITS).all(), "another layer was written"
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    assert hn.canaries_intact()


CASES = [
    # B, H, H_kv, T, lengths
    (5, 32, 8, 700, [700, 1, 333, 40, 9]),
    (3, 12, 2, 500, [500, 31, 257]),
    (2, 8, 8, 300, [300, 77]),
    (1, 8, 1, 3000, [3000]),
    (4, 14, 2, 200, [1, 2, 8, 200]),
]


@pytest.mark.parametrize("splits", [0, 1, 3, 152])
@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}_H{c[1]}_Hkv{c[2]}" for c in CASES])
def test_decode_over_int8_cache_matches_the_oracle(case, splits):
    B, H, H_kv, T, lengths = case
    hn = Q8Harness(1, B, H, H_kv, 128, T, seed=2200 + H + B)
    n_max = max(lengths)
    k, v = hn.rows(n_max, "fill")
    # append each sequence's live rows (cache_index 0, T_new = its length)
    for b, n in enumerate(lengths):
        ci = torch.zeros(B, dtype=torch.int32, device="cuda")
        kb = torch.zeros_like(k[:, :, :n]).copy_(k[:, :, :n])
        # append only sequence b: other sequences get an out-of-range index and are skipped
        ci.fill_(T + 1)
        ci[b] = 0
        assert hn.kvc.kvc_append(hn.h, 0, kb.contiguous(), v[:, :, :n].contiguous(), ci, n, None) == 0
    hn.kvc.kvc_get_error(hn.h, None)  # clears the index errors of the skipped sequences
    if splits:
        assert hn.kvc.kvc_set_num_splits(hn.h, splits) == 0
    q = hn.query("dec")
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
    vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_decode_attn(hn.h, 0, q, vl, n_max, out, None) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    _gpu.compare(out, _decode_ref(hn, 0, q, lengths), "bf16", "int8 decode")
    assert hn.canaries_intact()


def test_decode_steps_on_int8_cache():
    hn = Q8Harness(2, 3, 16, 4, 128, 400, seed=2300)
    pre = [0, 63, 390]
    for layer in range(2):
        k, v = hn.rows(max(pre), "pre", layer)
        for b, n in enumerate(pre):
            if n:
                ci = torch.full((3,), 401, dtype=torch.int32, device="cuda")
                ci[b] = 0
                assert hn.kvc.kvc_append(hn.h, layer, k[:, :, :n].contiguous(), v[:, :, :n].contiguous(), ci, n, None) == 0
    hn.kvc.kvc_get_error(hn.h, None)
    lengths = np.array(pre)
    for step in range(6):
        lengths = lengths + 1
        vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        for layer in range(2):
            k, v = hn.rows(1, "step", step, layer)
            q = hn.query("step", step, layer)
            out = torch.empty((3, 16, 128), dtype=torch.bfloat16, device="cuda")
            assert hn.kvc.kvc_decode_step(hn.h, layer, q, k, v, vl, int(lengths.max()), out, None) == 0
            torch.cuda.synchronize()
            _gpu.compare(out, _decode_ref(hn, layer, q, lengths), "bf16", f"int8 step {step} layer {layer}")
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    assert hn.canaries_intact()


# New rows at the interesting offsets of the int8 kernel's 128-row tiles:
# the first row, ends and starts of 8-row box groups and of tiles, the two
# 64-key halves of a tile, the last row of the buffer.
Q8_EDGE_LENGTHS = [1, 2, 8, 9, 63, 64, 65, 127, 128, 129, 136, 257, 511, 700]


def _fill_prefixes(hn, layer, pre, *tags):
    k, v = hn.rows(max(max(pre), 1), *tags)
    for b, n in enumerate(pre):
        if n:
            ci = torch.full((hn.B,), hn.T + 1, dtype=torch.int32, device="cuda")
            ci[b] = 0
            assert hn.kvc.kvc_append(hn.h, layer, k[:, :, :n].contiguous(), v[:, :, :n].contiguous(), ci, n,
                                     None) == 0
    hn.kvc.kvc_get_error(hn.h, None)   # the skipped sequences' index errors


@pytest.mark.parametrize("splits", [0, 1, 3, 13, 152])
def test_int8_fused_step_equals_append_then_decode(splits):
    """kvc_decode_step on an int8 cache quantises the new row inside the
    attention launch: the cache (codes and scales, padded rows included)
    equals kvc_append then kvc_decode_attn byte for byte, the new rows equal
    the oracle's quantisation, and the output matches the oracle."""
    B, T = len(Q8_EDGE_LENGTHS), 700
    lengths = np.array(Q8_EDGE_LENGTHS)
    fused, twice = Q8Harness(1, B, 16, 4, 128, T, seed=2700), Q8Harness(1, B, 16, 4, 128, T, seed=2700)
    for hn in (fused, twice):
        _fill_prefixes(hn, 0, (lengths - 1).tolist(), "pre")
        if splits:
            assert hn.kvc.kvc_set_num_splits(hn.h, splits) == 0
    kn, vn = fused.rows(1, "step")
    q = fused.query("step")
    vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out_f = torch.empty((B, 16, 128), dtype=torch.bfloat16, device="cuda")
    out_t = torch.empty_like(out_f)
    assert fused.kvc.kvc_decode_step(fused.h, 0, q, kn, vn, vl, T, out_f, None) == 0
    assert twice.kvc.kvc_append(twice.h, 0, kn, vn, vl - 1, 1, None) == 0
    assert twice.kvc.kvc_decode_attn(twice.h, 0, q, vl, T, out_t, None) == 0
    torch.cuda.synchronize()
    assert fused.kvc.kvc_get_error(fused.h, None) == 0 and twice.kvc.kvc_get_error(twice.h, None) == 0
    for a, b in ((fused.K, twice.K), (fused.V, twice.V), (fused.KS, twice.KS), (fused.VS, twice.VS)):
        assert torch.equal(a, b)
    kc, ks = quantize_rows(_gpu.bits(kn), "bf16")
    vc, vs = quantize_rows(_gpu.bits(vn), "bf16")
    for b, n in enumerate(lengths):
        assert np.array_equal(fused.K[0, b, :, n - 1].cpu().numpy(), kc[b, :, 0])
        assert np.array_equal(fused.V[0, b, :, n - 1].cpu().numpy(), vc[b, :, 0])
        assert np.array_equal(fused.KS[0, b, :, n - 1].cpu().numpy().view(np.float32), ks[b, :, 0])
        assert np.array_equal(fused.VS[0, b, :, n - 1].cpu().numpy().view(np.float32), vs[b, :, 0])
    ref = _decode_ref(fused, 0, q, lengths)
    _gpu.compare(out_f, ref, "bf16", "int8 fused step")
    _gpu.compare(out_t, ref, "bf16", "int8 append + decode")
    assert fused.canaries_intact() and twice.canaries_intact()


def test_int8_step_bad_valid_len_skips_append_and_output():
    hn = Q8Harness(1, 3, 8, 2, 128, 100, seed=2800)
    _fill_prefixes(hn, 0, [49, 10, 99], "bad")
    before = [t.clone() for t in (hn.K, hn.V, hn.KS, hn.VS)]
    kn, vn = hn.rows(1, "bad-step")
    q = hn.query("bad-step")
    for bad in (0, 101, -3):
        vl = torch.tensor([50, bad, 100], dtype=torch.int32, device="cuda")
        out = torch.full((3, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        assert hn.kvc.kvc_decode_step(hn.h, 0, q, kn, vn, vl, 100, out, None) == 0
        torch.cuda.synchronize()
        assert hn.kvc.kvc_get_error(hn.h, None) == hn.kvc.KVC_ERR_DEVICE_INDEX
        assert (out[1].float() == 7.0).all(), "a skipped sequence's output must stay unwritten"
        for t, t0 in zip((hn.K, hn.V, hn.KS, hn.VS), before):
            assert torch.equal(t[0, 1], t0[0, 1])
    ref = _decode_ref(hn, 0, q, np.array([50, 1, 100]))
    _gpu.compare(out[[0, 2]], ref[[0, 2]], "bf16", "the valid sequences")
    assert hn.canaries_intact()


def test_int8_attention_stays_close_to_the_unquantised_attention():
    """The quality side of section 4.4 ("a small quality cost"): on N(0,1)
    rows the int8 cache's attention output stays within 0.05 of the bf16
    cache's."""
    B, H, H_kv, T = 2, 16, 4, 600
    hn = Q8Harness(1, B, H, H_kv, 128, T, seed=2400)
    k, v = hn.rows(T, "cmp")
    assert hn.kvc.kvc_append(hn.h, 0, k, v, torch.zeros(B, dtype=torch.int32, device="cuda"), T, None) == 0
    q = hn.query("cmp")
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")
    vl = torch.full((B,), T, dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_decode_attn(hn.h, 0, q, vl, T, out, None) == 0
    torch.cuda.synchronize()
    ref16 = oracle.decode_attn(_gpu.bits(q), _gpu.bits(k), _gpu.bits(v), [T] * B, "bf16")
    err = np.abs(out.float().cpu().numpy() - ref16).max()
    assert err < 0.05, f"int8 vs bf16 cache: {err:.3e}"


def test_int8_host_errors():
    from static_kv_cache_gb300 import kvc
    cfg8 = kvc.make_config(1, 2, 8, 2, 128, 64, "int8")
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    ws = torch.empty(kvc.kvc_workspace_bytes(cfg8), dtype=torch.uint8, device="cuda")
    st, _ = kvc.kvc_alloc(cfg8, buf, buf, ws, ws.numel())
    assert st == kvc.KVC_ERR_INVALID, "kvc_alloc takes no int8 cache (scales missing)"
    st, _ = kvc.kvc_alloc_scaled(cfg8, buf, buf, 0, buf, ws, ws.numel())
    assert st == kvc.KVC_ERR_INVALID
    cfg16 = kvc.make_config(1, 2, 8, 2, 128, 64, "bf16")
    st, _ = kvc.kvc_alloc_scaled(cfg16, buf, buf, buf, buf, ws, ws.numel())
    assert st == kvc.KVC_ERR_INVALID
    assert kvc.kvc_check_config(kvc.make_config(1, 2, 8, 2, 64, 64, "int8")) == kvc.KVC_ERR_UNSUPPORTED
    assert kvc.kvc_scale_bytes(cfg16) == 0
    hn = Q8Harness(1, 2, 8, 2, 128, 64, seed=2500)
    q = hn.query("err")
    ci = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.empty((2, 8, 4, 128), dtype=torch.bfloat16, device="cuda")
    assert kvc.kvc_prefill_attn(hn.h, 0, q, ci, 4, out, None) == kvc.KVC_ERR_UNSUPPORTED
    vl = torch.ones(2, dtype=torch.int32, device="cuda")
    st = kvc.kvc_decode_attn_static(cfg8, 0, hn.kbuf.ptr(), hn.vbuf.ptr(), q, vl, 1, out, None)
    assert st == kvc.KVC_ERR_UNSUPPORTED


def test_int8_full_size_step_sampled():
    """The bench's int8 configuration: the Llama-3 layer (B=16, ragged
    U{1024..8192}) filled through the quantising append, one decode step;
    sampled sequences checked against the oracle over their dequantised rows."""
    w = synth.WORKLOADS["llama3_8b_int8"]
    lengths = synth.live_lengths(w).tolist()
    hn = Q8Harness(1, w.batch, w.n_heads, w.n_kv_heads, w.d_head, w.max_context, seed=2600)
    pre = [n - 1 for n in lengths]
    k, v = hn.rows(max(pre), "full-pre")
    for b, n in enumerate(pre):
        ci = torch.full((w.batch,), w.max_context + 1, dtype=torch.int32, device="cuda")
        ci[b] = 0
        assert hn.kvc.kvc_append(hn.h, 0, k[:, :, :n].contiguous(), v[:, :, :n].contiguous(), ci, n, None) == 0
    hn.kvc.kvc_get_error(hn.h, None)   # the skipped sequences' index errors
    kn, vn = hn.rows(1, "full-step")
    q = hn.query("full-step")
    vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = torch.empty((w.batch, w.n_heads, w.d_head), dtype=torch.bfloat16, device="cuda")
    assert hn.kvc.kvc_decode_step(hn.h, 0, q, kn, vn, vl, w.max_context, out, None) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    qd = oracle.widen(_gpu.bits(q), "bf16")
    for b in (0, 7, 15):
        n = lengths[b]
        codes_k = hn.K[0, b:b + 1, :, :n].cpu().numpy()
        codes_v = hn.V[0, b:b + 1, :, :n].cpu().numpy()
        sk = hn.KS[0, b:b + 1, :, :n].cpu().numpy().view(np.float32)
        sv = hn.VS[0, b:b + 1, :, :n].cpu().numpy().view(np.float32)
        ref = oracle.decode_attn(qd[b:b + 1], dequantize_rows(codes_k, sk), dequantize_rows(codes_v, sv),
                                 np.array([n]), "fp64")
        _gpu.compare(out[b:b + 1], ref, "bf16", f"int8 full size, sequence {b} (valid {n})")
    assert hn.canaries_intact()
