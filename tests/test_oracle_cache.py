"""The list-append cache: concatenation semantics, checked against a
pre-allocated buffer written by slice assignment ("KV Cache Optimization:
GQA Audit, In-Place Buffers, Persistent Prompts", #2 Before / After; the
page's smoke tests require both to give byte-identical output)."""
import numpy as np
import pytest

from oracle import ListAppendCache


def _rows(rng, B, H_kv, T, row_bytes):
    return rng.integers(0, 256, size=(B, H_kv, T, row_bytes), dtype=np.uint8)


def test_list_append_equals_slice_assign():
    rng = np.random.default_rng(0)
    L, B, H_kv, rb, cap = 2, 3, 2, 64, 100
    lc = ListAppendCache(L, B, H_kv, rb)
    buf_k = np.zeros((L, B, H_kv, cap, rb), np.uint8)
    buf_v = np.zeros_like(buf_k)
    valid = np.zeros((L, B), np.int64)
    for step, t_new in enumerate([64, 1, 1, 5, 1]):
        for layer in range(L):
            k, v = _rows(rng, B, H_kv, t_new, rb), _rows(rng, B, H_kv, t_new, rb)
            lc.append(layer, k, v, valid[layer], t_new)
            for b in range(B):
                s = valid[layer, b]
                buf_k[layer, b, :, s:s + t_new] = k[b]
                buf_v[layer, b, :, s:s + t_new] = v[b]
            valid[layer] += t_new
    for layer in range(L):
        for b in range(B):
            n = valid[layer, b]
            for kv in range(H_kv):
                assert lc.rows(layer, b, kv, "k") == buf_k[layer, b, kv, :n].tobytes()
                assert lc.rows(layer, b, kv, "v") == buf_v[layer, b, kv, :n].tobytes()


def test_prompt_then_single_steps_equals_one_append():
    """64 rows then 16 single rows == one append of the 80 rows."""
    rng = np.random.default_rng(1)
    B, H_kv, rb = 1, 8, 64
    k = _rows(rng, B, H_kv, 80, rb)
    v = _rows(rng, B, H_kv, 80, rb)
    a = ListAppendCache(1, B, H_kv, rb)
    a.append(0, k[:, :, :64], v[:, :, :64], [0], 64)
    for t in range(64, 80):
        a.append(0, k[:, :, t:t + 1], v[:, :, t:t + 1], [t], 1)
    b = ListAppendCache(1, B, H_kv, rb)
    b.append(0, k, v, [0], 80)
    for kv in range(H_kv):
        assert a.rows(0, 0, kv, "k") == b.rows(0, 0, kv, "k")
        assert a.rows(0, 0, kv, "v") == b.rows(0, 0, kv, "v")


def test_write_position_must_be_live_length():
    lc = ListAppendCache(1, 1, 1, 16)
    z = np.zeros((1, 1, 1, 16), np.uint8)
    lc.append(0, z, z, [0], 1)
    with pytest.raises(ValueError):
        lc.append(0, z, z, [3], 1)


def test_rewind_then_append_overwrites():
    """Rewind lowers the live length; the next append lands at the new end."""
    rng = np.random.default_rng(2)
    lc = ListAppendCache(1, 1, 1, 16)
    rows = _rows(rng, 1, 1, 6, 16)
    lc.append(0, rows[:, :, :5], rows[:, :, :5], [0], 5)
    lc.rewind(0, 0, 2)
    assert lc.length(0, 0) == 3
    lc.append(0, rows[:, :, 5:6], rows[:, :, 5:6], [3], 1)
    want = rows[0, 0, :3].tobytes() + rows[0, 0, 5].tobytes()
    assert lc.rows(0, 0, 0, "k") == want
