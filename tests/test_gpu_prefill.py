"""kvc_prefill_attn -- chunked-prefill attention over the static cache.

"KV-Cache Mechanics", AR Static KV-Cache: prefill fills the pre-allocated
cache from cache_index and decoding continues from there; "10.3", section 3:
the prompt's positions are processed together.  After a chunk of T_new rows
is appended at cache_index c, the query of chunk position t attends over
rows [0, c + t] (causal reading; see oracle/prefill.py).  Outputs are
compared with the fp64 oracle (bf16 / fp16 within 2e-2 absolute); rows past
a token's own position hold NaN poison, so reading one would show up as a
non-finite output.
"""
import numpy as np
import pytest
import torch

import oracle
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu


def _queries(w, T_new, *tags):
    return synth.normal((w.batch, w.n_heads, T_new, w.d_head), w.dtype,
                        synth.sub_seed(w.seed, "pq", T_new, *tags), device="cuda")


def _prefill(hn, layer, q, ci, T_new, out=None):
    w = hn.w
    if out is None:
        out = torch.empty((w.batch, w.n_heads, T_new, w.d_head), dtype=hn.tdtype, device="cuda")
    st = hn.kvc.kvc_prefill_attn(hn.h, layer, q, ci, T_new, out, None)
    return st, out


def _chunk(hn, layer, ci_list, T_new, *tags):
    """Append a chunk of T_new rows at ci and run the prefill attention;
    returns (q, out, K host bits, V host bits) for the oracle."""
    w = hn.w
    k, v = _gpu.new_rows(w, T_new, "chunk", *tags)
    ci = torch.tensor(ci_list, dtype=torch.int32, device="cuda")
    assert hn.append(layer, k, v, ci, T_new) == 0
    q = _queries(w, T_new, *tags)
    st, out = _prefill(hn, layer, q, ci, T_new)
    assert st == 0
    torch.cuda.synchronize()
    return q, out


def _expect(hn, layer, q, ci_list, T_new):
    Kh, Vh = _gpu.bits(hn.K[layer]), _gpu.bits(hn.V[layer])
    return oracle.prefill_attn(_gpu.bits(q), Kh, Vh, np.array(ci_list), T_new, hn.w.dtype)


def _compare(out, ref, dtype, what):
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output (a masked or padded row was read)"
    err = np.abs(got - ref).max()
    assert err <= 2e-2, f"{what}: max abs error {err:.3e}"
    return err


SHAPES = [
    # dtype, d_h, H, H_kv
    ("bf16", 128, 32, 8),
    ("bf16", 128, 8, 8),
    ("fp16", 64, 12, 2),
    ("bf16", 64, 16, 2),
    ("fp16", 128, 8, 1),
    ("bf16", 128, 6, 2),
]


@pytest.mark.parametrize("T_new", [1, 7, 16, 64, 100])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"{s[0]}_d{s[1]}_H{s[2]}_Hkv{s[3]}" for s in SHAPES])
def test_prompt_chunk_from_empty_cache(shape, T_new):
    dtype, D, H, H_kv = shape
    w = synth.Workload("pf_empty", 1, 2, H, H_kv, D, 160, dtype, steps=1, seed=1200 + D + H)
    hn = _gpu.Harness(w)
    q, out = _chunk(hn, 0, [0, 0], T_new, "empty")
    _compare(out, _expect(hn, 0, q, [0, 0], T_new), dtype, f"T_new={T_new}")
    assert hn.error() == 0 and hn.canaries_intact()


@pytest.mark.parametrize("shape", SHAPES[:3], ids=[f"{s[0]}_d{s[1]}_H{s[2]}_Hkv{s[3]}" for s in SHAPES[:3]])
def test_chunk_after_ragged_prefixes(shape):
    dtype, D, H, H_kv = shape
    pre = [0, 5, 31, 32, 250, 300]
    T_new = 45
    w = synth.Workload("pf_ragged", 1, len(pre), H, H_kv, D, 400, dtype, steps=1, seed=1300 + D)
    hn = _gpu.Harness(w)
    _gpu.fill_prefix(hn, 0, pre, "pre")
    q, out = _chunk(hn, 0, pre, T_new, "ragged")
    _compare(out, _expect(hn, 0, q, pre, T_new), dtype, "ragged prefixes")
    assert hn.error() == 0 and hn.canaries_intact()


def test_chunks_then_decode_steps_match_the_oracle():
    """A 96-token prompt as chunks of 40 and 56, then six decode steps, every
    output against the oracle over the cache as it stands."""
    w = synth.Workload("pf_flow", 2, 3, 16, 4, 128, 200, "bf16", steps=6, seed=1400)
    hn = _gpu.Harness(w)
    for layer in range(w.n_layers):
        pos = 0
        for T_new in (40, 56):
            q, out = _chunk(hn, layer, [pos] * w.batch, T_new, "flow", layer, pos)
            _compare(out, _expect(hn, layer, q, [pos] * w.batch, T_new), w.dtype, f"layer {layer} chunk at {pos}")
            pos += T_new
        for step in range(w.steps):
            valid = torch.full((w.batch,), pos + 1, dtype=torch.int32, device="cuda")
            k, v = _gpu.new_rows(w, 1, "flow-step", layer, step)
            qd = _gpu.query(w, "flow-step", layer, step)
            st, od = hn.step(layer, qd, k, v, valid, hint=pos + 1)
            assert st == 0
            Kh, Vh = _gpu.bits(hn.K[layer]), _gpu.bits(hn.V[layer])
            ref = oracle.decode_attn(_gpu.bits(qd), Kh, Vh, [pos + 1] * w.batch, w.dtype)
            _gpu.compare(od, ref, w.dtype, f"layer {layer} decode step {step}")
            pos += 1
    assert hn.error() == 0 and hn.canaries_intact()


def test_one_chunk_equals_two_chunks():
    """Processing a prompt in one chunk or in two gives the same rows."""
    w = synth.Workload("pf_split", 1, 2, 8, 2, 128, 128, "bf16", steps=1, seed=1500)
    one, two = _gpu.Harness(w), _gpu.Harness(w)
    k, v = _gpu.new_rows(w, 80, "split")
    q = _queries(w, 80, "split")
    zero = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert one.append(0, k, v, zero, 80) == 0
    st, out_one = _prefill(one, 0, q, zero, 80)
    assert st == 0
    thirty = torch.full((2,), 30, dtype=torch.int32, device="cuda")
    assert two.append(0, k[:, :, :30].contiguous(), v[:, :, :30].contiguous(), zero, 30) == 0
    st, out_a = _prefill(two, 0, q[:, :, :30].contiguous(), zero, 30)
    assert st == 0
    assert two.append(0, k[:, :, 30:].contiguous(), v[:, :, 30:].contiguous(), thirty, 50) == 0
    st, out_b = _prefill(two, 0, q[:, :, 30:].contiguous(), thirty, 50)
    assert st == 0
    torch.cuda.synchronize()
    both = torch.cat([out_a, out_b], dim=2)
    assert torch.equal(one.K.view(torch.uint8), two.K.view(torch.uint8))
    ref = _expect(one, 0, q, [0, 0], 80)
    _compare(out_one, ref, "bf16", "one chunk")
    _compare(both, ref, "bf16", "two chunks")


def test_bad_cache_index_is_reported_and_skipped():
    w = synth.Workload("pf_bad", 1, 3, 8, 2, 128, 100, "bf16", steps=1, seed=1600)
    hn = _gpu.Harness(w)
    T_new = 10
    _gpu.fill_prefix(hn, 0, [T_new, 0, 90 + T_new], "bad")  # prefix and chunk rows of the valid sequences
    q = _queries(w, T_new, "bad")
    for bad in (-1, 91, 200):
        ci = torch.tensor([0, bad, 90], dtype=torch.int32, device="cuda")
        out = torch.full((3, 8, T_new, 128), 3.0, dtype=torch.bfloat16, device="cuda")
        st, out = _prefill(hn, 0, q, ci, T_new, out=out)
        assert st == 0
        assert hn.error() == hn.kvc.KVC_ERR_DEVICE_INDEX
        assert (out[1].float() == 3.0).all()
    ref = _expect(hn, 0, q, [0, 0, 90], T_new)
    _compare(out[[0, 2]], ref[[0, 2]], "bf16", "valid sequences")


def test_prefill_host_errors():
    from static_kv_cache_gb300 import kvc
    w = synth.Workload("pf_err", 1, 2, 8, 2, 128, 64, "bf16", steps=1, seed=1700)
    hn = _gpu.Harness(w)
    q = _queries(w, 4, "err")
    ci = torch.zeros(2, dtype=torch.int32, device="cuda")
    out = torch.empty((2, 8, 4, 128), dtype=torch.bfloat16, device="cuda")
    assert kvc.kvc_prefill_attn(hn.h, 0, q, ci, 0, out, None) == kvc.KVC_OK
    assert kvc.kvc_prefill_attn(hn.h, 0, q, ci, 65, out, None) == kvc.KVC_ERR_CAPACITY
    assert kvc.kvc_prefill_attn(hn.h, 0, q, ci, -1, out, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_prefill_attn(hn.h, 1, q, ci, 4, out, None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_prefill_attn(hn.h, 0, q.data_ptr() + 2, ci, 4, out, None) == kvc.KVC_ERR_ALIGNMENT
    wf = synth.Workload("pf_f32", 1, 2, 8, 2, 128, 64, "fp32", steps=1, seed=1701)
    hf = _gpu.Harness(wf)
    qf = torch.zeros((2, 8, 4, 128), dtype=torch.float32, device="cuda")
    assert kvc.kvc_prefill_attn(hf.h, 0, qf, ci, 4, qf, None) == kvc.KVC_ERR_UNSUPPORTED
    assert hn.error() == 0


@pytest.mark.parametrize("prefixes", [None, [4096, 0, 4095, 31]], ids=["bench_prefixes", "longest_prefixes"])
def test_benchmarked_prefill_layer_against_the_oracle(prefixes):
    """One layer of the benchmarked chunked-prefill workload, in the launch
    configuration the benchmark times: Llama-3-8B-shaped cache (H=32, H_kv=8,
    d_h=128, bf16), B=4, a 512-token chunk each, after the workload's own
    live prefixes (drawn from U{0..4096}) and after the longest prefixes that
    range allows (4096 rows: the chunk's last CTAs stream 4608 key rows, over
    30 rounds of the ring of stages).  Every chunk row of sampled (sequence,
    KV head) groups -- one per sequence, two for the longest prefix -- is
    compared with the fp64 oracle element by element, and every output is
    checked finite."""
    w = synth.WORKLOADS["llama3_8b_prefill"].with_(n_layers=1)
    prefix = synth.live_lengths(w) if prefixes is None else torch.tensor(prefixes, dtype=torch.int32)
    T, g = w.chunk, w.group
    hn = _gpu.Harness(w)
    _gpu.fill_prefix(hn, 0, prefix.tolist(), "bench")
    q, out = _chunk(hn, 0, prefix.tolist(), T, "bench")
    assert hn.error() == 0 and hn.canaries_intact()
    assert torch.isfinite(out.float()).all(), "a masked or padded row was read"
    longest = int(np.argmax(prefix.numpy()))
    groups = [(b, (3 * b + 1) % w.n_kv_heads) for b in range(w.batch)] + [(longest, w.n_kv_heads - 1)]
    for b, kv in groups:
        ctx = int(prefix[b]) + T
        Kh = _gpu.bits(hn.K[0, b:b + 1, kv:kv + 1, :ctx])
        Vh = _gpu.bits(hn.V[0, b:b + 1, kv:kv + 1, :ctx])
        qh = _gpu.bits(q[b:b + 1, kv * g:(kv + 1) * g])
        ref = oracle.prefill_attn(qh, Kh, Vh, [int(prefix[b])], T, w.dtype)
        _compare(out[b:b + 1, kv * g:(kv + 1) * g], ref, w.dtype,
                 f"sequence {b} (prefix {int(prefix[b])}), KV head {kv}")
