"""A bounded wait inside the decode kernel runs out, and the handle recovers.

The split combine makes the last split of a (sequence, KV head) segment wait
for the partial results that the segment's other splits publish.  The test
makes that wait run out on purpose, from the host and without faulting
anything: before the launch it raises every arrival counter of the
caller-owned workspace far above the number of splits, so every split takes
a ticket that marks it as the segment's last one, none publishes, and each
waits for ready flags that nothing sets.  With the limit of that wait
shortened to a microsecond (kvc_set_wait_timeout_ns), every such wait gives
up at once: the kernel records KVC_ERR_TIMEOUT in the device error word and
the launch returns.  The copies into shared memory keep their 1 s limit and
finish.  kvc_get_error then reports the timeout and resets the counters, and
the next launch at the default limit matches the fp64 oracle.
"""
import pytest
import torch

import oracle
from static_kv_cache_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu

TICKETS_OFFSET = 256   # the workspace's arrival counters (documented in kvc.h)


def _case(seed):
    w = synth.Workload("timeout", 1, 3, 32, 8, 128, 2048, "bf16", steps=1, ragged=(1500, 2048), seed=seed)
    hn = _gpu.Harness(w)
    lengths = synth.live_lengths(w)
    _gpu.fill_prefix(hn, 0, (lengths - 1).tolist())
    torch.cuda.synchronize()
    k, v = _gpu.new_rows(w, 1, "t")
    q = _gpu.query(w, "t")
    maxlen = int(lengths.max())
    Kh = _gpu.bits(hn.K[0, :, :, :maxlen]).copy()
    Vh = _gpu.bits(hn.V[0, :, :, :maxlen]).copy()
    kb, vb = _gpu.bits(k), _gpu.bits(v)
    for b in range(w.batch):
        Kh[b, :, int(lengths[b]) - 1] = kb[b, :, 0]
        Vh[b, :, int(lengths[b]) - 1] = vb[b, :, 0]
    assert hn.append(0, k, v, (lengths - 1).cuda(), 1) == 0
    ref = oracle.decode_attn(_gpu.bits(q), Kh, Vh, lengths.numpy(), w.dtype)
    return w, hn, lengths, q, ref


def test_split_combine_wait_runs_out_and_the_handle_recovers():
    w, hn, lengths, q, ref = _case(61)
    kvc = hn.kvc
    valid = lengths.cuda()
    maxlen = int(lengths.max())
    segs = w.batch * w.n_kv_heads
    tickets = hn.wsbuf.data[TICKETS_OFFSET:TICKETS_OFFSET + 4 * segs].view(torch.int32)
    # 64 splits over 24 segments of 1500..2048 rows: every segment spans
    # several splits, so every piece goes through the split combine
    assert kvc.kvc_set_num_splits(hn.h, 64) == kvc.KVC_OK
    assert kvc.kvc_set_wait_timeout_ns(hn.h, 1000) == kvc.KVC_OK
    for _ in range(2):
        tickets.fill_(1 << 20)
        torch.cuda.synchronize()
        st, _ = hn.decode(0, q, valid, hint=maxlen)
        assert st == kvc.KVC_OK
        assert hn.error() == kvc.KVC_ERR_TIMEOUT
        assert int(tickets.abs().sum()) == 0, "kvc_get_error resets the counters after a timeout"
        assert hn.error() == kvc.KVC_OK, "the error word is cleared by the read"

    # back to the default limit: the same handle gives the right answer
    assert kvc.kvc_set_wait_timeout_ns(hn.h, 0) == kvc.KVC_OK
    for splits in (64, 0):
        assert kvc.kvc_set_num_splits(hn.h, splits) == kvc.KVC_OK
        st, out = hn.decode(0, q, valid, hint=maxlen)
        assert st == kvc.KVC_OK
        _gpu.compare(out, ref, w.dtype, f"after the timeout, splits={splits}")
        assert hn.error() == kvc.KVC_OK
    assert hn.canaries_intact()


def test_short_limit_without_injection_is_either_clean_or_a_reported_timeout():
    """A 1 us limit on an ordinary launch: the splits may or may not publish
    in time; either the output is right and no error is recorded, or the
    timeout is reported -- never a wrong answer without an error."""
    w, hn, lengths, q, ref = _case(62)
    kvc = hn.kvc
    valid = lengths.cuda()
    assert kvc.kvc_set_num_splits(hn.h, 64) == kvc.KVC_OK
    assert kvc.kvc_set_wait_timeout_ns(hn.h, 1000) == kvc.KVC_OK
    for _ in range(3):
        st, out = hn.decode(0, q, valid, hint=int(lengths.max()))
        assert st == kvc.KVC_OK
        e = hn.error()
        assert e in (kvc.KVC_OK, kvc.KVC_ERR_TIMEOUT)
        if e == kvc.KVC_OK:
            _gpu.compare(out, ref, w.dtype, "1 us limit, no timeout recorded")
    assert kvc.kvc_set_wait_timeout_ns(hn.h, 0) == kvc.KVC_OK
    st, out = hn.decode(0, q, valid, hint=int(lengths.max()))
    assert st == kvc.KVC_OK
    _gpu.compare(out, ref, w.dtype, "default limit")
    assert hn.error() == kvc.KVC_OK and hn.canaries_intact()
