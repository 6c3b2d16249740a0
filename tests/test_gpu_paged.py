"""Paged caches on the GPU ("10.3 -- KV cache implementation details",
section 7, PagedAttention: 16-token blocks made logically contiguous by a
block table; the layout reading is in oracle/paged.py).

Pools [L, num_blocks, H_kv, 16, d_h] hold NaN everywhere no live row was
written, so a read of a padded row or of an unused block shows up as a
non-finite output.  Checked: decode through random tables against the fp64
oracle over oracle.paged.gather; blocks shared by two sequences; the append
writing through the table (bit-exact with the list cache); fused decode steps;
a table entry out of range; host errors.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import ListAppendCache, paged
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


class PagedHarness:
    def __init__(self, L, B, H, H_kv, D, T, dtype, num_blocks, seed, share_first=0):
        from static_kv_cache_gb300 import kvc
        self.kvc, self.L, self.B, self.H, self.H_kv, self.D, self.T = kvc, L, B, H, H_kv, D, T
        self.dtype, self.seed, self.num_blocks = dtype, seed, num_blocks
        self.tdt = synth.DTYPES[dtype]
        self.cfg = kvc.make_config(L, B, H, H_kv, D, T, dtype)
        nbytes = kvc.kvc_pool_bytes(self.cfg, num_blocks)
        assert nbytes == L * num_blocks * H_kv * 16 * D * synth.ELEM_BYTES[dtype]
        self.kbuf, self.vbuf = _gpu.Guarded(nbytes), _gpu.Guarded(nbytes)
        shape = (L, num_blocks, H_kv, 16, D)
        self.K = self.kbuf.view(self.tdt, shape)
        self.V = self.vbuf.view(self.tdt, shape)
        synth.poison_(self.K, dtype)
        synth.poison_(self.V, dtype)
        mb = T // 16
        perm = np.random.default_rng(seed).permutation(num_blocks)
        table = perm[:B * mb].reshape(B, mb).astype(np.int32)
        if share_first:  # sequence 1 reads sequence 0's first blocks
            table[1, :share_first] = table[0, :share_first]
        self.table_host = table
        self.tbuf = _gpu.Guarded(table.nbytes)
        self.table = self.tbuf.view(torch.int32, table.shape)
        self.table.copy_(torch.from_numpy(table))
        self.ws = _gpu.Guarded(kvc.kvc_workspace_bytes(self.cfg))
        st, self.h = kvc.kvc_alloc_paged(self.cfg, self.kbuf.ptr(), self.vbuf.ptr(), num_blocks, self.tbuf.ptr(),
                                         self.ws.ptr(), self.ws.nbytes)
        kvc.check(st, "kvc_alloc_paged")

    def rows(self, T_new, *tags):
        shape = (self.B, self.H_kv, T_new, self.D)
        return (synth.normal(shape, self.dtype, synth.sub_seed(self.seed, "pk", *tags), device="cuda"),
                synth.normal(shape, self.dtype, synth.sub_seed(self.seed, "pv", *tags), device="cuda"))

    def query(self, *tags):
        return synth.normal((self.B, self.H, self.D), self.dtype, synth.sub_seed(self.seed, "pq", *tags), device="cuda")

    def dense(self, layer, ctx):
        """The logical rows through the oracle's gather (bits)."""
        kp, vp = _gpu.bits(self.K[layer]), _gpu.bits(self.V[layer])
        return paged.gather(kp, self.table_host, ctx), paged.gather(vp, self.table_host, ctx)

    def fill(self, layer, lengths, *tags):
        """Append rows [0, lengths[b]) of every sequence through the library."""
        n_max = max(lengths)
        k, v = self.rows(n_max, "fill", layer, *tags)
        for b, n in enumerate(lengths):
            if n == 0:
                continue
            ci = torch.full((self.B,), self.T + 1, dtype=torch.int32, device="cuda")   # others skipped
            ci[b] = 0
            assert self.kvc.kvc_append(self.h, layer, k[:, :, :n].contiguous(), v[:, :, :n].contiguous(), ci, n, None) == 0
        self.kvc.kvc_get_error(self.h, None)   # the skipped sequences' index errors
        return k, v

    def canaries_intact(self):
        return all(b.canaries_intact() for b in (self.kbuf, self.vbuf, self.tbuf, self.ws))


CASES = [
    # dtype, D, H, H_kv, B, T, lengths
    ("bf16", 128, 32, 8, 5, 704, [704, 1, 333, 40, 17]),
    ("fp16", 128, 12, 2, 3, 400, [400, 9, 255]),
    ("fp16", 64, 12, 2, 3, 512, [512, 31, 257]),
    ("bf16", 128, 16, 2, 2, 1600, [1600, 15]),
    ("bf16", 64, 8, 1, 1, 2048, [2048]),
    ("bf16", 128, 32, 1, 3, 800, [800, 17, 401]),
    ("fp16", 64, 32, 2, 2, 512, [512, 100]),
    # 2 or 4 query heads per KV head and an even H_kv: the kernel that reads a
    # block two KV heads at a time; an odd H_kv keeps one head per tile
    ("fp16", 64, 8, 4, 3, 512, [512, 31, 257]),
    ("bf16", 128, 12, 6, 2, 400, [17, 400]),
    ("bf16", 128, 12, 3, 3, 320, [320, 1, 129]),
]


@pytest.mark.parametrize("splits", [0, 1, 3, 152])
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_d{c[1]}_H{c[2]}_Hkv{c[3]}_B{c[4]}" for c in CASES])
def test_paged_decode_matches_the_oracle(case, splits):
    dtype, D, H, H_kv, B, T, lengths = case
    hn = PagedHarness(1, B, H, H_kv, D, T, dtype, num_blocks=B * (T // 16) + 7, seed=3100 + D + H)
    hn.fill(0, lengths)
    if splits:
        assert hn.kvc.kvc_set_num_splits(hn.h, splits) == 0
    q = hn.query("dec")
    vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = torch.empty((B, H, D), dtype=hn.tdt, device="cuda")
    assert hn.kvc.kvc_decode_attn(hn.h, 0, q, vl, max(lengths), out, None) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    Kd, Vd = hn.dense(0, max(lengths))
    _gpu.compare(out, oracle.decode_attn(_gpu.bits(q), Kd, Vd, np.array(lengths), dtype), dtype, "paged decode")
    assert hn.canaries_intact()


def test_blocks_shared_between_sequences():
    hn = PagedHarness(1, 2, 16, 4, 128, 256, "bf16", num_blocks=40, seed=3200, share_first=3)
    # sequence 0 writes 48 rows (3 blocks) that sequence 1 also maps; sequence 1 then continues alone
    k, v = hn.rows(48, "share")
    ci = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_append(hn.h, 0, k, v, ci, 48, None) == 0
    hn.kvc.kvc_get_error(hn.h, None)
    k2, v2 = hn.rows(20, "tail")
    ci = torch.tensor([300, 48], dtype=torch.int32, device="cuda")
    assert hn.kvc.kvc_append(hn.h, 0, k2, v2, ci, 20, None) == 0
    hn.kvc.kvc_get_error(hn.h, None)
    q = hn.query("share")
    vl = torch.tensor([48, 68], dtype=torch.int32, device="cuda")
    out = torch.empty((2, 16, 128), dtype=torch.bfloat16, device="cuda")
    assert hn.kvc.kvc_decode_attn(hn.h, 0, q, vl, 68, out, None) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    Kd, Vd = hn.dense(0, 68)
    _gpu.compare(out, oracle.decode_attn(_gpu.bits(q), Kd, Vd, np.array([48, 68]), "bf16"), "bf16", "shared blocks")
    # the shared rows are sequence 0's
    assert np.array_equal(Kd[1, :, :48], Kd[0, :, :48])


@pytest.mark.parametrize("dtype,D,H,H_kv", [("bf16", 128, 16, 4), ("fp16", 64, 6, 2), ("fp16", 64, 8, 4)])
def test_paged_decode_steps_and_append_through_the_table(dtype, D, H, H_kv):
    B, T, L = 3, 256, 2
    hn = PagedHarness(L, B, H, H_kv, D, T, dtype, num_blocks=B * (T // 16) + 3, seed=3300 + D)
    lc = ListAppendCache(L, B, H_kv, D * synth.ELEM_BYTES[dtype])
    pre = [0, 15, 200]
    for layer in range(L):
        k, v = hn.fill(layer, pre, "pre")
        kb, vb = _gpu.bits(k), _gpu.bits(v)
        for b, n in enumerate(pre):
            for kv in range(H_kv):
                for t in range(n):
                    lc.k[layer][b][kv].append(kb[b, kv, t].view(np.uint8).tobytes())
                    lc.v[layer][b][kv].append(vb[b, kv, t].view(np.uint8).tobytes())
    lengths = np.array(pre)
    for step in range(5):
        ci = lengths.copy()
        lengths = lengths + 1
        vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
        for layer in range(L):
            k, v = hn.rows(1, "step", step, layer)
            q = hn.query("step", step, layer)
            out = torch.empty((B, H, D), dtype=hn.tdt, device="cuda")
            assert hn.kvc.kvc_decode_step(hn.h, layer, q, k, v, vl, int(lengths.max()), out, None) == 0
            lc.append(layer, _gpu.bits(k), _gpu.bits(v), ci, 1)
            ctx = int(lengths.max())
            ref = oracle.decode_attn(_gpu.bits(q), lc.dense(layer, "k", ctx).view(np.uint16),
                                     lc.dense(layer, "v", ctx).view(np.uint16), lengths, dtype)
            _gpu.compare(out, ref, dtype, f"paged step {step} layer {layer}")
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    for layer in range(L):   # the pools hold exactly the list cache's rows, through the table
        Kd, Vd = hn.dense(layer, int(lengths.max()))
        kd, vd = lc.dense(layer, "k", int(lengths.max())).view(np.uint16), lc.dense(layer, "v", int(lengths.max())).view(np.uint16)
        for b in range(B):
            n = int(lengths[b])
            assert np.array_equal(Kd[b, :, :n].view(np.uint16), kd[b, :, :n])
            assert np.array_equal(Vd[b, :, :n].view(np.uint16), vd[b, :, :n])
    assert hn.canaries_intact()


def test_bad_table_entry_is_reported_without_a_fault():
    hn = PagedHarness(1, 2, 8, 2, 128, 128, "bf16", num_blocks=20, seed=3400)
    hn.fill(0, [40, 40])
    hn.table[1, 1] = 999          # out of range
    q = hn.query("bad")
    vl = torch.tensor([40, 40], dtype=torch.int32, device="cuda")
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    assert hn.kvc.kvc_decode_attn(hn.h, 0, q, vl, 40, out, None) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == hn.kvc.KVC_ERR_DEVICE_INDEX
    Kd, Vd = hn.dense(0, 40)      # sequence 0 is unaffected
    _gpu.compare(out[:1], oracle.decode_attn(_gpu.bits(q)[:1], Kd[:1], Vd[:1], np.array([40]), "bf16"), "bf16", "good sequence")
    k, v = hn.rows(1, "bad-append")
    assert hn.kvc.kvc_append(hn.h, 0, k, v, torch.tensor([40, 20], dtype=torch.int32, device="cuda"), 1, None) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == hn.kvc.KVC_ERR_DEVICE_INDEX
    assert hn.canaries_intact()


def test_paged_host_errors():
    from static_kv_cache_gb300 import kvc
    buf = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    tab = torch.zeros(64, dtype=torch.int32, device="cuda")
    def alloc(cfg, nb=10, t=tab):
        ws = torch.empty(max(1, kvc.kvc_workspace_bytes(cfg)), dtype=torch.uint8, device="cuda")
        return kvc.kvc_alloc_paged(cfg, buf, buf, nb, t, ws, ws.numel())[0]
    assert alloc(kvc.make_config(1, 2, 8, 8, 128, 64, "bf16")) == kvc.KVC_ERR_UNSUPPORTED    # g = 1: CUDA-core kernel
    assert alloc(kvc.make_config(1, 2, 8, 2, 128, 64, "fp32")) == kvc.KVC_ERR_UNSUPPORTED
    assert alloc(kvc.make_config(1, 2, 8, 2, 128, 64, "int8")) == kvc.KVC_ERR_UNSUPPORTED
    assert alloc(kvc.make_config(1, 2, 8, 2, 128, 60, "bf16")) == kvc.KVC_ERR_INVALID        # not a multiple of 16
    assert alloc(kvc.make_config(1, 2, 8, 2, 128, 64, "bf16"), nb=0) == kvc.KVC_ERR_INVALID
    hn = PagedHarness(1, 2, 8, 2, 128, 64, "bf16", num_blocks=10, seed=3500)
    q = torch.empty((2, 8, 4, 128), dtype=torch.bfloat16, device="cuda")
    ci = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert kvc.kvc_prefill_attn(hn.h, 0, q, ci, 4, q, None) == kvc.KVC_ERR_UNSUPPORTED


def test_paged_full_size_sampled():
    """The bench's paged configuration: the Llama-3 layer (B=16, ragged
    U{1024..8192}) in 16-row blocks under a random table, one fused step;
    sampled sequences checked against the oracle over the gathered rows."""
    w = synth.WORKLOADS["llama3_8b_paged"]
    lengths = synth.live_lengths(w).tolist()
    hn = PagedHarness(1, w.batch, w.n_heads, w.n_kv_heads, w.d_head, w.max_context, w.dtype,
                      num_blocks=w.batch * (w.max_context // 16) + 5, seed=3600)
    hn.fill(0, [n - 1 for n in lengths], "full")
    k, v = hn.rows(1, "full-step")
    q = hn.query("full-step")
    vl = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    out = torch.empty((w.batch, w.n_heads, w.d_head), dtype=hn.tdt, device="cuda")
    assert hn.kvc.kvc_decode_step(hn.h, 0, q, k, v, vl, w.max_context, out) == 0
    assert hn.kvc.kvc_get_error(hn.h, None) == 0
    kp, vp = _gpu.bits(hn.K[0]), _gpu.bits(hn.V[0])
    for b in (0, 5, 11, 15):
        n = lengths[b]
        Kd = paged.gather(kp, hn.table_host[b:b + 1], n)
        Vd = paged.gather(vp, hn.table_host[b:b + 1], n)
        assert np.array_equal(Kd[0, :, n - 1], _gpu.bits(k)[b, :, 0]), "new row written through the table"
        ref = oracle.decode_attn(_gpu.bits(q)[b:b + 1], Kd, Vd, np.array([n]), w.dtype)
        _gpu.compare(out[b:b + 1], ref, w.dtype, f"paged full size, sequence {b} (valid {n})")
    assert hn.canaries_intact()
