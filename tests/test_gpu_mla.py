"""MLA latent-cache decode on the GPU against the fp64 oracle.

"10.3 -- KV cache implementation details", section 4.3: one cached latent
per token, keys and values rebuilt per head by up-projections
(oracle.mla_decode_attn writes that definition out).  The GPU takes the
absorbed order; its only roundings beyond fp32 accumulation are the absorbed
query and the attended latent (once each, to the cache type, as tensor-core
operands), the probabilities fed to the tensor-core product (bf16 / fp16,
each in [0, 1]), and the output (once).

Checked: decode over ragged lengths and several split counts for every
compiled (d_c, H) with both 16-bit types; a step sequence whose cache bytes
equal a list-append cache bit for bit; multi-row appends; a full-size
sampled case; out-of-range lengths; host refusals.  Latent rows past the live
length hold NaN, so any read of them that reaches the arithmetic shows.

Bar: the decode tolerance of 2e-2 absolute for 16-bit outputs, and, because
the outputs of a diffuse softmax are small, also 2e-2 of the largest |ref| of
each (b, h) row.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import ListAppendCache
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


def mla_compare(got, ref, what):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    assert err.max() <= 2e-2, f"{what}: max abs error {err.max():.3e}"
    rel = (err / np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)).max()
    assert rel <= 2e-2, f"{what}: error {rel:.3e} of the row max"
    return err.max(), rel


class MlaHarness:
    def __init__(self, L, B, H, d_h, d_c, T, dtype, seed, q_scale=1.0):
        from static_kv_cache_gb300 import kvc
        self.kvc, self.L, self.B, self.H, self.d_h, self.d_c, self.T = kvc, L, B, H, d_h, d_c, T
        self.dtype, self.seed, self.q_scale = dtype, seed, q_scale
        self.tdt = synth.DTYPES[dtype]
        self.cfg = kvc.make_mla_config(L, B, H, d_h, d_c, T, dtype)
        nbytes = kvc.kvc_mla_cache_bytes(self.cfg)
        assert nbytes == L * B * T * d_c * 2
        self.cbuf = _gpu.Guarded(nbytes)
        self.C = self.cbuf.view(self.tdt, (L, B, T, d_c))
        synth.poison_(self.C, dtype)
        self.ws = _gpu.Guarded(kvc.kvc_mla_workspace_bytes(self.cfg))
        self.ws.data.zero_()
        st, self.h = kvc.kvc_mla_alloc(self.cfg, self.cbuf.ptr(), self.ws.ptr(), self.ws.nbytes)
        kvc.check(st, "kvc_mla_alloc")
        # up-projections: entries N(0, 1/d_c), so rebuilt rows have unit variance
        self.wk = (synth.normal((H, d_h, d_c), "fp32", synth.sub_seed(seed, "wk"), device="cuda")
                   / d_c ** 0.5).to(self.tdt)
        self.wv = (synth.normal((H, d_h, d_c), "fp32", synth.sub_seed(seed, "wv"), device="cuda")
                   / d_c ** 0.5).to(self.tdt)

    def latents(self, T_new, *tags):
        return synth.normal((self.B, T_new, self.d_c), self.dtype, synth.sub_seed(self.seed, "c", *tags), device="cuda")

    def query(self, *tags):
        q = synth.normal((self.B, self.H, self.d_h), "fp32", synth.sub_seed(self.seed, "q", *tags), device="cuda")
        return (q * self.q_scale).to(self.tdt)

    def fill(self, layer, lengths, *tags):
        """Rows [0, lengths[b]) through kvc_mla_append, one call per sequence."""
        c = self.latents(max(lengths), "fill", layer, *tags)
        for b, n in enumerate(lengths):
            if n == 0:
                continue
            ci = torch.full((self.B,), self.T + 1, dtype=torch.int32, device="cuda")
            ci[b] = 0
            assert self.kvc.kvc_mla_append(self.h, layer, c[:, :n].contiguous(), ci, n) == 0
        self.kvc.kvc_mla_get_error(self.h)   # the skipped sequences' index errors
        return c

    def decode(self, layer, q, lengths, hint=0):
        vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        out = torch.empty((self.B, self.H, self.d_h), dtype=self.tdt, device="cuda")
        assert self.kvc.kvc_mla_decode_attn(self.h, layer, q, self.wk, self.wv, vl, hint, out) == 0
        return out

    def reference(self, layer, q, lengths):
        ctx = max(lengths)
        return oracle.mla_decode_attn(_gpu.bits(q), _gpu.bits(self.C[layer, :, :ctx]), _gpu.bits(self.wk),
                                      _gpu.bits(self.wv), np.array(lengths), self.dtype)

    def canaries_intact(self):
        return self.cbuf.canaries_intact() and self.ws.canaries_intact()


SHAPES = [  # dtype, H, d_h, d_c
    ("bf16", 16, 128, 512), ("fp16", 16, 128, 512), ("bf16", 8, 64, 512),
    ("bf16", 16, 64, 256), ("fp16", 8, 128, 256), ("bf16", 16, 128, 128), ("bf16", 8, 32, 128),
    # more than 16 heads: the 16-head kernel over head groups ("10.3" §4.3:
    # every head attends over the same latent rows)
    ("bf16", 32, 128, 512), ("fp16", 48, 64, 256), ("bf16", 128, 128, 512),
]


@pytest.mark.parametrize("splits", [0, 1, 3, 152])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}_H{s[1]}_dh{s[2]}_dc{s[3]}" for s in SHAPES])
def test_mla_decode_matches_the_oracle(shape, splits):
    dtype, H, d_h, d_c = shape
    lengths = [700, 1, 63, 64, 65, 129, 333]
    hn = MlaHarness(1, len(lengths), H, d_h, d_c, 704, dtype, seed=4000 + H + d_c)
    hn.fill(0, lengths)
    if splits:
        assert hn.kvc.kvc_mla_set_num_splits(hn.h, splits) == 0
    q = hn.query("dec")
    out = hn.decode(0, q, lengths)
    assert hn.kvc.kvc_mla_get_error(hn.h) == 0
    mla_compare(out, hn.reference(0, q, lengths), f"mla {shape} splits {splits}")
    assert hn.canaries_intact()


@pytest.mark.parametrize("B,d_h", [(70, 128), (5, 256), (17, 16)])
def test_mla_batch_and_head_width_edges(B, d_h):
    """More than 64 sequences (a second absorb block), and the narrowest and
    widest head widths the kernels take."""
    lengths = [(37 * b) % 300 + 1 for b in range(B)]
    hn = MlaHarness(1, B, 16, d_h, 256, 304, "bf16", seed=4600 + B + d_h)
    hn.fill(0, lengths)
    q = hn.query("edge")
    out = hn.decode(0, q, lengths)
    assert hn.kvc.kvc_mla_get_error(hn.h) == 0
    mla_compare(out, hn.reference(0, q, lengths), f"B={B} d_h={d_h}")
    assert hn.canaries_intact()


@pytest.mark.parametrize("q_scale", [4.0])
def test_mla_peaky_attention(q_scale):
    lengths = [300, 41, 512]
    hn = MlaHarness(1, 3, 16, 128, 512, 512, "bf16", seed=4100, q_scale=q_scale)
    hn.fill(0, lengths)
    q = hn.query("peaky")
    out = hn.decode(0, q, lengths)
    ref = hn.reference(0, q, lengths)
    assert np.abs(ref).max() > 0.5, "peaky case should give O(1) outputs"
    mla_compare(out, ref, "peaky")


@pytest.mark.parametrize("dtype,H,d_h,d_c", [("bf16", 16, 128, 512), ("fp16", 8, 64, 256)])
def test_mla_step_sequence_and_cache_bytes(dtype, H, d_h, d_c):
    B, T, L, steps = 4, 300, 2, 5
    hn = MlaHarness(L, B, H, d_h, d_c, T, dtype, seed=4200 + d_c)
    lc = ListAppendCache(L, B, 1, d_c * 2)
    pre = [0, 17, 64, 250]
    for layer in range(L):
        c = hn.fill(layer, pre, "pre")
        cb = _gpu.bits(c)
        for b, n in enumerate(pre):
            for t in range(n):
                lc.k[layer][b][0].append(cb[b, t].view(np.uint8).tobytes())
    lengths = np.array(pre)
    for step in range(steps):
        ci = lengths.copy()
        lengths = lengths + 1
        vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        for layer in range(L):
            c_new = hn.latents(1, "step", step, layer)
            q = hn.query("step", step, layer)
            out = torch.empty((B, H, d_h), dtype=hn.tdt, device="cuda")
            assert hn.kvc.kvc_mla_decode_step(hn.h, layer, q, c_new, hn.wk, hn.wv, vl, int(lengths.max()), out) == 0
            cb = _gpu.bits(c_new)[:, None]          # [B, 1 (head), 1, d_c]
            lc.append(layer, cb, cb, ci, 1)
            ctx = int(lengths.max())
            ref = oracle.mla_decode_attn(_gpu.bits(q), lc.dense(layer, "k", ctx).view(np.uint16)[:, 0],
                                         _gpu.bits(hn.wk), _gpu.bits(hn.wv), lengths, dtype)
            mla_compare(out, ref, f"step {step} layer {layer}")
    assert hn.kvc.kvc_mla_get_error(hn.h) == 0
    poison = synth.POISON_BITS[dtype]
    for layer in range(L):
        got = _gpu.bits(hn.C[layer])
        want = lc.dense(layer, "k", int(lengths.max())).view(np.uint16)[:, 0]
        for b in range(B):
            n = int(lengths[b])
            assert np.array_equal(got[b, :n], want[b, :n]), f"latent rows of sequence {b}"
            assert (got[b, n] == poison).all(), "the row after the live ones stays untouched"
    assert hn.canaries_intact()


@pytest.mark.parametrize("splits", [1, 3, 152])
@pytest.mark.parametrize("H", [16, 32])
def test_mla_steps_with_forced_splits(splits, H):
    """Fused steps whose new rows fall at every position of a 64-row tile
    (the first, the last, across a tile edge), under forced splits: the
    attention launch copies the tiles without a new row before its
    dependency wait and the new-row tiles after it; outputs against the
    oracle, the cache bytes against a list-append cache."""
    B, T, L, steps = 7, 300, 1, 3
    hn = MlaHarness(L, B, H, 128, 512, T, "bf16", seed=4700 + splits + H)
    assert hn.kvc.kvc_mla_set_num_splits(hn.h, splits) == 0
    lc = ListAppendCache(L, B, 1, 512 * 2)
    pre = [0, 1, 62, 63, 64, 127, 200]
    c = hn.fill(0, pre, "pre")
    cb = _gpu.bits(c)
    for b, n in enumerate(pre):
        for t in range(n):
            lc.k[0][b][0].append(cb[b, t].view(np.uint8).tobytes())
    lengths = np.array(pre)
    for step in range(steps):
        ci = lengths.copy()
        lengths = lengths + 1
        vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        c_new = hn.latents(1, "fstep", step)
        q = hn.query("fstep", step)
        out = torch.empty((B, H, 128), dtype=hn.tdt, device="cuda")
        assert hn.kvc.kvc_mla_decode_step(hn.h, 0, q, c_new, hn.wk, hn.wv, vl, int(lengths.max()), out) == 0
        cnb = _gpu.bits(c_new)[:, None]
        lc.append(0, cnb, cnb, ci, 1)
        ctx = int(lengths.max())
        ref = oracle.mla_decode_attn(_gpu.bits(q), lc.dense(0, "k", ctx).view(np.uint16)[:, 0],
                                     _gpu.bits(hn.wk), _gpu.bits(hn.wv), lengths, "bf16")
        mla_compare(out, ref, f"step {step} splits {splits} H {H}")
    assert hn.kvc.kvc_mla_get_error(hn.h) == 0
    got = _gpu.bits(hn.C[0])
    want = lc.dense(0, "k", int(lengths.max())).view(np.uint16)[:, 0]
    for b in range(B):
        n = int(lengths[b])
        assert np.array_equal(got[b, :n], want[b, :n]), f"latent rows of sequence {b}"
    assert hn.canaries_intact()


def test_mla_multi_row_append_is_bit_exact():
    hn = MlaHarness(2, 3, 8, 64, 256, 200, "bf16", seed=4300)
    c = hn.latents(50, "multi")
    ci = torch.tensor([0, 30, 150], dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_mla_append(hn.h, 1, c, ci, 50) == 0
    assert hn.kvc.kvc_mla_get_error(hn.h) == 0
    got, cb = _gpu.bits(hn.C[1]), _gpu.bits(c)
    for b, start in enumerate([0, 30, 150]):
        assert np.array_equal(got[b, start:start + 50], cb[b])
    assert (_gpu.bits(hn.C[0]) == synth.POISON_BITS["bf16"]).all(), "other layer untouched"
    bad = torch.tensor([0, 151, 10], dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_mla_append(hn.h, 0, c, bad, 50) == 0
    assert hn.kvc.kvc_mla_get_error(hn.h) == hn.kvc.KVC_ERR_DEVICE_INDEX
    assert hn.canaries_intact()


def test_mla_bad_lengths_skip_the_sequence():
    lengths = [40, 40, 40]
    hn = MlaHarness(1, 3, 16, 128, 512, 64, "bf16", seed=4400)
    hn.fill(0, lengths)
    q = hn.query("bad")
    for bad in (0, 65, -2):
        vl = torch.tensor([40, bad, 40], dtype=torch.int32, device="cuda")
        out = torch.full((3, 16, 128), 7.0, device="cuda").to(torch.bfloat16)
        assert hn.kvc.kvc_mla_decode_attn(hn.h, 0, q, hn.wk, hn.wv, vl, 64, out) == 0
        assert hn.kvc.kvc_mla_get_error(hn.h) == hn.kvc.KVC_ERR_DEVICE_INDEX
        assert (out[1].float() == 7.0).all(), "a skipped sequence's output stays unwritten"
        ref = hn.reference(0, q, lengths)
        mla_compare(out[[0, 2]], ref[[0, 2]], f"valid sequences next to length {bad}")
    assert hn.canaries_intact()


def test_mla_full_size_sampled():
    """The bench's latent cache shape (B = 64, H = 16, d_h = 128, d_c = 512,
    ragged lengths U{1024..8192}), one layer, all sequences decoded in one
    launch; sampled sequences checked against the oracle."""
    w = synth.WORKLOADS["mla_dsv2"]
    lengths = synth.live_lengths(w).tolist()
    hn = MlaHarness(1, w.batch, w.n_heads, w.d_head, w.d_latent, w.max_context, w.dtype, seed=4500)
    for b in range(w.batch):    # rows drawn directly (the prefill's state), then one step through the library
        n = lengths[b] - 1
        hn.C[0, b, :n] = synth.normal((n, w.d_latent), w.dtype, synth.sub_seed(4500, "pc", b), device="cuda")
    c_new = hn.latents(1, "full")[:, 0].contiguous()
    q = hn.query("full")
    vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = torch.empty((w.batch, w.n_heads, w.d_head), dtype=hn.tdt, device="cuda")
    assert hn.kvc.kvc_mla_decode_step(hn.h, 0, q, c_new, hn.wk, hn.wv, vl, w.max_context, out) == 0
    assert hn.kvc.kvc_mla_get_error(hn.h) == 0
    for b in (0, 17, 40, 63):
        n = lengths[b]
        ref = oracle.mla_decode_attn(_gpu.bits(q[b:b + 1]), _gpu.bits(hn.C[0, b:b + 1, :n]), _gpu.bits(hn.wk),
                                     _gpu.bits(hn.wv), np.array([n]), w.dtype)
        mla_compare(out[b:b + 1], ref, f"sequence {b} (valid {n})")


def test_mla_host_errors():
    from static_kv_cache_gb300 import kvc
    buf = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    ws = torch.empty(kvc.kvc_mla_workspace_bytes(kvc.make_mla_config(1, 2, 16, 128, 512, 64, "bf16")),
                     dtype=torch.uint8, device="cuda")
    def alloc(*shape):
        cfg = kvc.make_mla_config(*shape)
        return kvc.kvc_mla_alloc(cfg, buf, ws, ws.numel())[0]
    assert alloc(1, 2, 16, 128, 96, 64, "bf16") == kvc.KVC_ERR_UNSUPPORTED     # d_c not compiled
    assert alloc(1, 2, 24, 128, 512, 64, "bf16") == kvc.KVC_ERR_UNSUPPORTED    # H not a multiple of 16
    assert alloc(1, 2, 144, 128, 512, 64, "bf16") == kvc.KVC_ERR_UNSUPPORTED   # H above 128
    assert alloc(1, 2, 16, 128, 512, 64, "fp32") == kvc.KVC_ERR_UNSUPPORTED
    assert alloc(1, 2, 16, 0, 512, 64, "bf16") == kvc.KVC_ERR_INVALID
    cfg = kvc.make_mla_config(1, 2, 16, 128, 512, 64, "bf16")
    assert kvc.kvc_mla_alloc(cfg, buf, ws, 100)[0] == kvc.KVC_ERR_WORKSPACE
    assert kvc.kvc_mla_alloc(cfg, buf.data_ptr() + 2, ws, ws.numel())[0] == kvc.KVC_ERR_ALIGNMENT
    st, h = kvc.kvc_mla_alloc(cfg, buf, ws, ws.numel())
    assert st == 0
    q = torch.zeros((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((16, 128, 512), dtype=torch.bfloat16, device="cuda")
    vl = torch.ones(2, dtype=torch.int32, device="cuda")
    assert kvc.kvc_mla_decode_attn(h, 1, q, w, w, vl, 1, q) == kvc.KVC_ERR_INVALID       # layer
    assert kvc.kvc_mla_decode_attn(h, 0, q, w, w, vl, 65, q) == kvc.KVC_ERR_INVALID      # hint
    assert kvc.kvc_mla_decode_attn(h, 0, q.data_ptr() + 2, w, w, vl, 1, q) == kvc.KVC_ERR_ALIGNMENT
    assert kvc.kvc_mla_decode_step(h, 0, q, None, w, w, vl, 1, q) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_mla_append(h, 0, q, vl, 65) == kvc.KVC_ERR_CAPACITY
    assert kvc.kvc_mla_get_error(h) == 0
    kvc.kvc_mla_free(h)
