"""The fp64 attention oracle against references that are not itself."""
import pytest

from tests import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(oracle_lib, pin):
    pin(oracle_lib)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_library_sdpa_all_dtypes(oracle_lib, dtype):
    _pins.pin_library_sdpa(oracle_lib, dtype=dtype)


@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 1), (12, 2), (6, 3)])
def test_library_sdpa_groupings(oracle_lib, H, H_kv):
    """MHA (g = 1), MQA (H_kv = 1, "10.3", section 4.1) and GQA groupings."""
    _pins.pin_library_sdpa(oracle_lib, H=H, H_kv=H_kv, d=16, ctx=33)


def test_poisoned_rows_are_not_read(oracle_lib):
    """Rows at or past the live length ("KV Cache Optimization...", #2: reads
    are sliced to validLengths) do not influence the result."""
    import numpy as np
    import oracle
    from static_kv_cache_gb300 import synth
    q, K, V = _pins._inputs("bf16", 2, 4, 2, 16, 30, 5)
    valid = np.array([9, 30], np.int32)
    clean = oracle.decode_attn(q, K, V, valid, "bf16", lib=oracle_lib)
    K2, V2 = K.copy(), V.copy()
    K2[0, :, 9:] = synth.POISON_BITS["bf16"]
    V2[0, :, 9:] = synth.POISON_BITS["bf16"]
    poisoned = oracle.decode_attn(q, K2, V2, valid, "bf16", lib=oracle_lib)
    assert np.array_equal(clean, poisoned)


def test_rejects_bad_lengths(oracle_lib):
    import numpy as np
    import oracle
    q, K, V = _pins._inputs("fp32", 1, 2, 1, 8, 4, 3)
    for bad in (0, 5, -1):
        with pytest.raises(ValueError):
            oracle.decode_attn(q, K, V, np.array([bad], np.int32), "fp32", lib=oracle_lib)
