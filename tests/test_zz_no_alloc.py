"""kvc_decode_attn_static: decode attention without any device allocation.

Some callers cannot call cudaMalloc or hand the library a workspace -- their
device memory belongs to a host framework or plugin interface that passes only
the tensors of each call.  For them the library offers an entry point that
keeps its scratch in an array compiled into the library.  These tests check,
through the C ABI and on two calls in a row, that its output matches the fp64
oracle and the regular entry point (which uses a caller-owned workspace);
that the one-CTA-per-segment launch of small problems and a skipped sequence
work; that device-side errors reach the array's own error word; and that a
configuration too large for the array is refused.

This file is collected last, so a run that stops at the first failure has
run every other test before it.
"""
import pytest
import torch

import oracle
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


def _drain_error_word(kvc):
    """The array's error word is shared by every call on the device and keeps
    the first error until read; start each test from a clear word."""
    kvc.kvc_static_get_error(None)


def _static_calls(kvc, cfg, layer, hn, q, valid, hint, like, n=2):
    outs = []
    for _ in range(n):                      # calls in a row share the array
        out = torch.full_like(like, float("nan"))
        st = kvc.kvc_decode_attn_static(cfg, layer, hn.kbuf.ptr(), hn.vbuf.ptr(), q, valid, hint, out, None)
        assert st == kvc.KVC_OK
        outs.append(out)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("dtype,H,H_kv", [("bf16", 32, 8), ("fp32", 12, 2)])
def test_static_scratch_matches_oracle_and_workspace_entry_point(dtype, H, H_kv):
    w = synth.Workload(f"noalloc_{dtype}", 2, 5, H, H_kv, 128, 3000, dtype, steps=1,
                       ragged=(1, 3000), seed=777)
    hn = _gpu.Harness(w)
    kvc = hn.kvc
    _drain_error_word(kvc)
    lengths = synth.live_lengths(w)
    lengths[0] = w.max_context
    lengths[1] = 1
    layer = 1
    _gpu.fill_prefix(hn, layer, (lengths - 1).tolist())
    k, v = _gpu.new_rows(w, 1, "na")
    q = _gpu.query(w, "na")
    valid = lengths.cuda()
    assert hn.append(layer, k, v, (lengths - 1).cuda(), 1) == 0
    maxlen = int(lengths.max())
    torch.cuda.synchronize()
    ref = oracle.decode_attn(_gpu.bits(q), _gpu.bits(hn.K[layer, :, :, :maxlen]),
                             _gpu.bits(hn.V[layer, :, :, :maxlen]), lengths.numpy(), dtype)

    st, regular = hn.decode(layer, q, valid, hint=maxlen)
    assert st == 0
    assert hn.error() == 0

    for out in _static_calls(kvc, hn.cfg, layer, hn, q, valid, maxlen, regular):
        _gpu.compare(out, ref, dtype, "static scratch vs the oracle")
        err = (out.float() - regular.float()).abs().max().item()
        if dtype == "fp32":
            assert err <= 1e-5 * regular.float().abs().max().item()
        else:
            assert err <= 2e-2
    assert kvc.kvc_static_get_error(None) == kvc.KVC_OK
    assert hn.canaries_intact()


def test_static_scratch_small_problem_and_skipped_sequence():
    """B * H_kv below the SM count and short segments: the launch takes one
    CTA per (sequence, KV head).  One sequence has valid_len 0: the call
    succeeds, that sequence's rows stay unwritten, the others match the
    oracle, and the array's error word reports the bad length once."""
    w = synth.Workload("noalloc_small", 1, 6, 8, 2, 32, 256, "bf16", steps=1, ragged=(1, 256), seed=778)
    hn = _gpu.Harness(w)
    kvc = hn.kvc
    _drain_error_word(kvc)
    lengths = synth.live_lengths(w)
    lengths[2] = 256
    _gpu.fill_prefix(hn, 0, lengths.tolist())
    q = _gpu.query(w, "small")
    torch.cuda.synchronize()
    maxlen = int(lengths.max())
    ref = oracle.decode_attn(_gpu.bits(q), _gpu.bits(hn.K[0, :, :, :maxlen]),
                             _gpu.bits(hn.V[0, :, :, :maxlen]), lengths.numpy(), "bf16")
    like = torch.empty((w.batch, w.n_heads, w.d_head), dtype=torch.bfloat16, device="cuda")
    for out in _static_calls(kvc, hn.cfg, 0, hn, q, lengths.cuda(), maxlen, like):
        _gpu.compare(out, ref, "bf16", "small problem")
    assert kvc.kvc_static_get_error(None) == kvc.KVC_OK

    bad = lengths.clone()
    bad[4] = 0
    good = [b for b in range(w.batch) if b != 4]
    for out in _static_calls(kvc, hn.cfg, 0, hn, q, bad.cuda(), maxlen, like):
        assert torch.isnan(out[4].float()).all(), "a skipped sequence's rows stay unwritten"
        _gpu.compare(out[good], ref[good], "bf16", "the other sequences")
    assert kvc.kvc_static_get_error(None) == kvc.KVC_ERR_DEVICE_INDEX
    assert kvc.kvc_static_get_error(None) == kvc.KVC_OK
    assert hn.canaries_intact()


def test_static_scratch_refuses_too_large_configs():
    from static_kv_cache_gb300 import kvc
    cfg = kvc.make_config(1, 256, 64, 8, 256, 64, "bf16")   # needs ~18 MB of split partials
    dummy = torch.empty(4096, dtype=torch.uint8, device="cuda")
    vl = torch.ones(256, dtype=torch.int32, device="cuda")
    st = kvc.kvc_decode_attn_static(cfg, 0, dummy, dummy, dummy, vl, 1, dummy, None)
    assert st == kvc.KVC_ERR_WORKSPACE
