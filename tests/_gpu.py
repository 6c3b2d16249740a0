"""GPU-side test harness: caller-owned buffers with guard canaries, poisoned
caches, and the calls through the C ABI.

Inputs come from ``static_kv_cache_gb300.synth``; expected values come only
from ``oracle``.  Nothing here computes attention.
"""
from __future__ import annotations

import numpy as np
import torch

from static_kv_cache_gb300 import synth

GUARD = 4096          # canary bytes before and after every buffer
ALIGN = 256


class Guarded:
    """A device byte buffer with canary regions on both sides."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = nbytes
        self.raw = torch.empty(GUARD + nbytes + GUARD + ALIGN, dtype=torch.uint8, device=device)
        self.raw.fill_(synth.CANARY_BYTE)
        base = self.raw.data_ptr()
        pad = (-(base + GUARD)) % ALIGN
        self.off = GUARD + pad
        self.data = self.raw[self.off:self.off + nbytes]

    def ptr(self) -> int:
        return self.data.data_ptr()

    def canaries_intact(self) -> bool:
        before = self.raw[:self.off]
        after = self.raw[self.off + self.nbytes:]
        return bool((before == synth.CANARY_BYTE).all()) and bool((after == synth.CANARY_BYTE).all())

    def view(self, dtype, shape):
        return self.data.view(dtype).view(*shape)


class Harness:
    """One static cache [L, B, H_kv, T_max, D] for K and V, a workspace, and
    a kvc handle bound to them."""

    def __init__(self, w: synth.Workload, poison: bool = True):
        from static_kv_cache_gb300 import kvc
        self.kvc = kvc
        self.w = w
        self.tdtype = synth.DTYPES[w.dtype]
        self.eb = synth.ELEM_BYTES[w.dtype]
        self.shape = (w.n_layers, w.batch, w.n_kv_heads, w.max_context, w.d_head)
        nbytes = int(np.prod(self.shape)) * self.eb
        self.kbuf = Guarded(nbytes)
        self.vbuf = Guarded(nbytes)
        self.K = self.kbuf.view(self.tdtype, self.shape)
        self.V = self.vbuf.view(self.tdtype, self.shape)
        if poison:
            synth.poison_(self.K, w.dtype)
            synth.poison_(self.V, w.dtype)
        self.cfg = kvc.make_config(w.n_layers, w.batch, w.n_heads, w.n_kv_heads, w.d_head,
                                   w.max_context, w.dtype)
        self.ws_bytes = kvc.kvc_workspace_bytes(self.cfg)
        self.wsbuf = Guarded(self.ws_bytes)
        st, self.h = kvc.kvc_alloc(self.cfg, self.kbuf.ptr(), self.vbuf.ptr(), self.wsbuf.ptr(),
                                   self.ws_bytes)
        kvc.check(st, "kvc_alloc")

    def close(self):
        if self.h is not None:
            self.kvc.kvc_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- calls through the C ABI
    def append(self, layer, k_new, v_new, cache_index, T_new, stream=None):
        return self.kvc.kvc_append(self.h, layer, k_new, v_new, cache_index, T_new, stream)

    def decode(self, layer, q, valid_len, hint=0, out=None, stream=None):
        w = self.w
        if out is None:
            out = torch.empty((w.batch, w.n_heads, w.d_head), dtype=self.tdtype, device="cuda")
        st = self.kvc.kvc_decode_attn(self.h, layer, q, valid_len, hint, out, stream)
        return st, out

    def step(self, layer, q, k_new, v_new, valid_len, hint=0, out=None, stream=None):
        w = self.w
        if out is None:
            out = torch.empty((w.batch, w.n_heads, w.d_head), dtype=self.tdtype, device="cuda")
        st = self.kvc.kvc_decode_step(self.h, layer, q, k_new, v_new, valid_len, hint, out, stream)
        return st, out

    def error(self, stream=None):
        return self.kvc.kvc_get_error(self.h, stream)

    def canaries_intact(self) -> bool:
        return (self.kbuf.canaries_intact() and self.vbuf.canaries_intact()
                and self.wsbuf.canaries_intact())


def new_rows(w: synth.Workload, T_new: int, *tags):
    shape = (w.batch, w.n_kv_heads, T_new, w.d_head)
    k = synth.normal(shape, w.dtype, synth.sub_seed(w.seed, "k_new", *tags), device="cuda")
    v = synth.normal(shape, w.dtype, synth.sub_seed(w.seed, "v_new", *tags), device="cuda")
    return k, v


def query(w: synth.Workload, *tags):
    return synth.normal((w.batch, w.n_heads, w.d_head), w.dtype,
                        synth.sub_seed(w.seed, "q", *tags), device="cuda")


def fill_prefix(hn: Harness, layer: int, lengths, *tags):
    """Write N(0,1) rows [0, lengths[b]) of one layer directly with torch (the
    state a prefill leaves behind), before any kernel of the library runs on
    that layer."""
    w = hn.w
    for b in range(w.batch):
        n = int(lengths[b])
        if n == 0:
            continue
        shape = (w.n_kv_heads, n, w.d_head)
        hn.K[layer, b, :, :n] = synth.normal(shape, w.dtype, synth.sub_seed(w.seed, "pk", layer, b, *tags),
                                             device="cuda")
        hn.V[layer, b, :, :n] = synth.normal(shape, w.dtype, synth.sub_seed(w.seed, "pv", layer, b, *tags),
                                             device="cuda")


def bits(t: torch.Tensor):
    return synth.to_bits(t)


def compare(got: torch.Tensor, ref: np.ndarray, dtype: str, what: str = ""):
    """The parity bar: bf16 / fp16 outputs within 2e-2 absolute of the fp64
    oracle; fp32 outputs within 1e-5 of the largest |ref| of each (b, h) row."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    if dtype == "fp32":
        scale = np.abs(ref).max(axis=-1, keepdims=True)
        rel = (err / np.maximum(scale, 1e-30)).max()
        assert rel <= 1e-5, f"{what}: fp32 error {rel:.3e} of the row max"
        return rel
    worst = err.max()
    assert worst <= 2e-2, f"{what}: {dtype} max abs error {worst:.3e}"
    return worst
