"""kvc_decode_attn_static: decode attention without any device allocation.

Some callers cannot call cudaMalloc or hand the library a workspace -- their
device memory belongs to a host framework or plugin interface that passes only
the tensors of each call.  For them the library offers an entry point that
keeps its scratch in an array compiled into the library.  These tests check,
through the C ABI, that two calls in a row give the same output as the
regular entry point (which uses a caller-owned workspace), and that a
configuration too large for the array is refused.
"""
import pytest
import torch

from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,H,H_kv", [("bf16", 32, 8), ("fp32", 12, 2)])
def test_static_scratch_matches_workspace_entry_point(dtype, H, H_kv):
    w = synth.Workload(f"noalloc_{dtype}", 2, 5, H, H_kv, 128, 3000, dtype, steps=1,
                       ragged=(1, 3000), seed=777)
    hn = _gpu.Harness(w)
    kvc = hn.kvc
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

    st, ref = hn.decode(layer, q, valid, hint=maxlen)
    assert st == 0
    assert hn.error() == 0

    outs = []
    for _ in range(2):                      # two calls in a row share the array
        out = torch.full_like(ref, float("nan"))
        st = kvc.kvc_decode_attn_static(hn.cfg, layer, hn.kbuf.ptr(), hn.vbuf.ptr(), q, valid,
                                        maxlen, out, None)
        assert st == kvc.KVC_OK
        outs.append(out)
    torch.cuda.synchronize()
    for out in outs:
        assert torch.isfinite(out.float()).all()
        err = (out.float() - ref.float()).abs().max().item()
        if dtype == "fp32":
            assert err <= 1e-5 * ref.float().abs().max().item()
        else:
            assert err <= 2e-2
    assert hn.canaries_intact()


def test_static_scratch_refuses_too_large_configs():
    from static_kv_cache_gb300 import kvc
    cfg = kvc.make_config(1, 256, 64, 8, 256, 64, "bf16")   # needs ~18 MB of split partials
    dummy = torch.empty(4096, dtype=torch.uint8, device="cuda")
    vl = torch.ones(256, dtype=torch.int32, device="cuda")
    st = kvc.kvc_decode_attn_static(cfg, 0, dummy, dummy, dummy, vl, 1, dummy, None)
    assert st == kvc.KVC_ERR_WORKSPACE
