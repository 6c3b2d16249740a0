"""Pins of the int8-cache oracle (oracle.quantize_rows / dequantize_rows).

"10.3 -- KV cache implementation details", section 4.4: the cache may be
stored as int8 (p = 1).  The scheme is a reading (symmetric, one fp32 scale
per row, codes rint(x * 127 / absmax) in fp32; see oracle/quant.py).  Pinned
by rows worked out by hand, the error bound of round-to-nearest on a
127-step grid, the exact +-127 code of each row's largest element, a
lossless case where int8 attention must equal the unquantised attention
exactly, and planted mistakes.
"""
import numpy as np
import pytest

import oracle
from oracle import dequantize_rows, quantize_rows


def test_rows_worked_by_hand():
    # [1, -2, 0.5, 0]: absmax 2, 127/2 = 63.5 exactly; 1*63.5 = 63.5 -> 64
    # (half to even), -2*63.5 = -127, 0.5*63.5 = 31.75 -> 32, 0 -> 0.
    codes, scale = quantize_rows(np.array([[1.0, -2.0, 0.5, 0.0]], dtype=np.float32), "fp32")
    assert codes.tolist() == [[64, -127, 32, 0]]
    assert scale[0] == np.float32(2.0) / np.float32(127.0)
    # [0.5, -0.25]: 127/0.5 = 254; 0.5*254 = 127, -0.25*254 = -63.5 -> -64.
    codes, scale = quantize_rows(np.array([[0.5, -0.25]], dtype=np.float32), "fp32")
    assert codes.tolist() == [[127, -64]]
    # a row of zeros: scale 0, codes 0
    codes, scale = quantize_rows(np.zeros((1, 8), dtype=np.float32), "fp32")
    assert (codes == 0).all() and scale[0] == 0.0


def _rows(n, d, dtype, seed):
    gen = np.random.default_rng(seed)
    x = (gen.standard_normal((n, d)) * gen.uniform(0.01, 30, size=(n, 1))).astype(np.float32)
    if dtype == "fp32":
        return x
    if dtype == "bf16":
        u = x.view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return x.astype(np.float16).view(np.uint16)


def _invariants(x_bits, dtype, quant=quantize_rows):
    x = oracle.widen(x_bits, dtype)
    codes, scale = quant(x_bits, dtype)
    xh = dequantize_rows(codes, scale)
    s = scale.astype(np.float64)[:, None]
    ok_range = bool((np.abs(codes.astype(np.int32)) <= 127).all())
    err_bound = bool((np.abs(x - xh) <= 0.5 * s * (1 + 1e-5) + 1e-30).all())
    top = bool((np.abs(codes.astype(np.int32)).max(axis=1) == 127).all())
    sign = bool(((np.sign(codes) == np.sign(x)) | (codes == 0)).all())
    return ok_range and err_bound and top and sign


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_invariants_on_random_rows(dtype):
    assert _invariants(_rows(500, 128, dtype, seed=3), dtype)


def test_lossless_rows_give_the_unquantised_attention():
    """Rows of the form k/8 with integer |k| <= 127 and a +-127 in every row
    quantise without loss (scale 1/8), so int8 attention must equal the
    attention over the original bf16 rows exactly."""
    gen = np.random.default_rng(11)
    B, H, H_kv, d, n = 2, 8, 2, 64, 40
    k_int = gen.integers(-127, 128, size=(B, H_kv, n, d))
    v_int = gen.integers(-127, 128, size=(B, H_kv, n, d))
    k_int[..., 0] = 127
    v_int[..., 3] = -127
    K = (k_int / 8.0).astype(np.float32)
    V = (v_int / 8.0).astype(np.float32)
    kc, ks = quantize_rows(K, "fp32")
    vc, vs = quantize_rows(V, "fp32")
    assert (ks == np.float32(127.0 / 8.0) / np.float32(127.0)).all()
    assert np.array_equal(kc, k_int.astype(np.int8)) and np.array_equal(vc, v_int.astype(np.int8))
    q = gen.standard_normal((B, H, d)).astype(np.float32)
    valid = np.array([n, 17])
    ref = oracle.decode_attn(q, K, V, valid, "fp32")
    got = oracle.decode_attn(q.astype(np.float64), dequantize_rows(kc, ks), dequantize_rows(vc, vs), valid, "fp64")
    assert np.array_equal(got, ref)


# ---- planted mistakes ------------------------------------------------------
def _q_scale_128(x_bits, dtype):
    x = oracle.widen(x_bits, dtype).astype(np.float32)
    am = np.abs(x).max(axis=-1)
    scale = (am / np.float32(128.0)).astype(np.float32)
    codes = np.clip(np.rint(x * (np.float32(128.0) / am)[..., None]), -127, 127).astype(np.int8)
    return codes, scale


def _q_floor(x_bits, dtype):
    x = oracle.widen(x_bits, dtype).astype(np.float32)
    am = np.abs(x).max(axis=-1)
    scale = (am / np.float32(127.0)).astype(np.float32)
    codes = np.clip(np.floor(x * (np.float32(127.0) / am)[..., None]), -127, 127).astype(np.int8)
    return codes, scale


def _q_per_tensor(x_bits, dtype):
    x = oracle.widen(x_bits, dtype).astype(np.float32)
    am = np.float32(np.abs(x).max())
    codes = np.clip(np.rint(x * (np.float32(127.0) / am)), -127, 127).astype(np.int8)
    return codes, np.full(x.shape[:-1], am / np.float32(127.0), dtype=np.float32)


@pytest.mark.parametrize("mutant", [_q_scale_128, _q_floor, _q_per_tensor],
                         ids=["scale_absmax_over_128", "floor_not_round", "one_scale_per_tensor"])
def test_planted_mistakes_break_the_invariants(mutant):
    assert not _invariants(_rows(200, 128, "bf16", seed=5), "bf16", quant=mutant)
