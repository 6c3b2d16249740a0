"""In-place append on the GPU, bit-exact against the list-append oracle.

"KV Cache Optimization: GQA Audit, In-Place Buffers, Persistent Prompts",
#2: slice-assigning into the pre-allocated buffer must reproduce the
concatenating cache byte for byte; rows past the live length and memory
outside the buffers must stay untouched.
"""
import numpy as np
import pytest
import torch

from oracle import ListAppendCache
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


def _poison_u8(dtype, row_bytes):
    bitsv = synth.POISON_BITS[dtype]
    if dtype == "fp32":
        return np.frombuffer(np.array([bitsv] * (row_bytes // 4), np.uint32).tobytes(), np.uint8)
    return np.frombuffer(np.array([bitsv] * (row_bytes // 2), np.uint16).tobytes(), np.uint8)


def _check_cache_equals_list(hn, lc, layer):
    w = hn.w
    Kh = hn.K[layer].contiguous().view(torch.uint8).cpu().numpy()  # [B, H_kv, T_max, row_bytes]
    Vh = hn.V[layer].contiguous().view(torch.uint8).cpu().numpy()
    poison = _poison_u8(w.dtype, w.row_bytes)
    for b in range(w.batch):
        n = lc.length(layer, b)
        for kv in range(w.n_kv_heads):
            assert Kh[b, kv, :n].tobytes() == lc.rows(layer, b, kv, "k"), (layer, b, kv)
            assert Vh[b, kv, :n].tobytes() == lc.rows(layer, b, kv, "v"), (layer, b, kv)
            assert (Kh[b, kv, n:] == poison).all() and (Vh[b, kv, n:] == poison).all(), \
                f"rows past the live length were written (layer {layer}, b {b})"


@pytest.mark.parametrize("name", ["tiny_mha", "small_gqa"])
def test_append_sequence_bit_exact(name):
    w = synth.WORKLOADS[name]
    hn = _gpu.Harness(w)
    lc = ListAppendCache(w.n_layers, w.batch, w.n_kv_heads, w.row_bytes)
    first = w.first_append or w.prefill
    for layer in range(w.n_layers):
        k, v = _gpu.new_rows(w, first, "first", layer)
        ci = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
        assert hn.append(layer, k, v, ci, first) == 0
        lc.append(layer, _gpu.bits(k), _gpu.bits(v), [0] * w.batch, first)
    for step in range(w.steps):
        pos = first + step
        ci = torch.full((w.batch,), pos, dtype=torch.int32, device="cuda")
        for layer in range(w.n_layers):
            k, v = _gpu.new_rows(w, 1, step, layer)
            assert hn.append(layer, k, v, ci, 1) == 0
            lc.append(layer, _gpu.bits(k), _gpu.bits(v), [pos] * w.batch, 1)
    assert hn.error() == 0
    for layer in range(w.n_layers):
        _check_cache_equals_list(hn, lc, layer)
    assert hn.canaries_intact()


def test_append_ragged_positions():
    """Different write positions per sequence in one call."""
    w = synth.Workload("ragged_append", 2, 5, 8, 4, 64, 300, "bf16", steps=1, seed=77)
    hn = _gpu.Harness(w)
    lc = ListAppendCache(w.n_layers, w.batch, w.n_kv_heads, w.row_bytes)
    lengths = [0, 3, 17, 250, 295]          # 295 + 1 + 4 = max_context
    for layer in range(w.n_layers):
        _gpu.fill_prefix(hn, layer, lengths)
        for b, n in enumerate(lengths):
            kb = _gpu.bits(hn.K[layer, b, :, :n]).view(np.uint8).reshape(w.n_kv_heads, n, w.row_bytes)
            vb = _gpu.bits(hn.V[layer, b, :, :n]).view(np.uint8).reshape(w.n_kv_heads, n, w.row_bytes)
            for kv in range(w.n_kv_heads):
                for t in range(n):
                    lc.k[layer][b][kv].append(kb[kv, t].tobytes())
                    lc.v[layer][b][kv].append(vb[kv, t].tobytes())
    ci_host = list(lengths)
    for T_new in (1, 4):
        ci = torch.tensor(ci_host, dtype=torch.int32, device="cuda")
        for layer in range(w.n_layers):
            k, v = _gpu.new_rows(w, T_new, "rag", T_new, layer)
            assert hn.append(layer, k, v, ci, T_new) == 0
            lc.append(layer, _gpu.bits(k), _gpu.bits(v), ci_host, T_new)
        ci_host = [c + T_new for c in ci_host]
    assert hn.error() == 0
    for layer in range(w.n_layers):
        _check_cache_equals_list(hn, lc, layer)
    assert hn.canaries_intact()


@pytest.mark.parametrize("dtype,d", [("fp32", 128), ("fp16", 64), ("bf16", 256), ("fp32", 32)])
def test_append_dtypes_and_widths(dtype, d):
    w = synth.Workload(f"app_{dtype}_{d}", 1, 3, 4, 2, d, 100, dtype, steps=1, seed=5)
    hn = _gpu.Harness(w)
    lc = ListAppendCache(1, w.batch, w.n_kv_heads, w.row_bytes)
    pos = 0
    for T_new in (7, 1, 33, 1):
        k, v = _gpu.new_rows(w, T_new, T_new, pos)
        ci = torch.full((w.batch,), pos, dtype=torch.int32, device="cuda")
        assert hn.append(0, k, v, ci, T_new) == 0
        lc.append(0, _gpu.bits(k), _gpu.bits(v), [pos] * w.batch, T_new)
        pos += T_new
    assert hn.error() == 0
    _check_cache_equals_list(hn, lc, 0)
    assert hn.canaries_intact()


def test_append_device_index_out_of_range_is_reported_and_skipped():
    w = synth.Workload("bad_index", 1, 3, 4, 2, 64, 50, "bf16", steps=1, seed=9)
    hn = _gpu.Harness(w)
    before_k = hn.K.clone()
    k, v = _gpu.new_rows(w, 2, "bad")
    # sequence 0 fine, sequence 1 passes the end, sequence 2 negative
    ci = torch.tensor([10, 49, -1], dtype=torch.int32, device="cuda")
    assert hn.append(0, k, v, ci, 2) == 0
    assert hn.error() == hn.kvc.KVC_ERR_DEVICE_INDEX
    assert hn.error() == 0, "the error word is cleared by reading it"
    after = hn.K
    assert torch.equal(after[0, 1].view(torch.int16), before_k[0, 1].view(torch.int16))
    assert torch.equal(after[0, 2].view(torch.int16), before_k[0, 2].view(torch.int16))
    assert torch.equal(after[0, 0, :, 10:12].view(torch.int16), k[0].view(torch.int16))
    assert hn.canaries_intact()


def test_append_host_errors():
    w = synth.Workload("host_err", 2, 2, 4, 2, 64, 32, "bf16", steps=1, seed=3)
    hn = _gpu.Harness(w)
    kvc = hn.kvc
    k, v = _gpu.new_rows(w, 1, "h")
    ci = torch.zeros(w.batch, dtype=torch.int32, device="cuda")
    assert hn.append(2, k, v, ci, 1) == kvc.KVC_ERR_INVALID          # layer out of range
    assert hn.append(-1, k, v, ci, 1) == kvc.KVC_ERR_INVALID
    big_k, big_v = _gpu.new_rows(w, 33, "big")
    assert hn.append(0, big_k, big_v, ci, 33) == kvc.KVC_ERR_CAPACITY
    assert hn.append(0, None, v, ci, 1) == kvc.KVC_ERR_INVALID
    raw = torch.empty(k.numel() * 2 + 16, dtype=torch.uint8, device="cuda")
    assert hn.append(0, raw.data_ptr() + 2, v, ci, 1) == kvc.KVC_ERR_ALIGNMENT
    assert hn.append(0, k, v, ci, 0) == kvc.KVC_OK                   # no-op
    assert hn.error() == 0
    assert hn.canaries_intact()
