"""The cache-size formula against every figure the pages print for it."""
import os

import pytest

from oracle import formula

HERE = os.path.dirname(os.path.abspath(__file__))
UNITS = {"B": 1, "GB": 10**9, "MB": 10**6, "GiB": 2**30, "MiB": 2**20}


def _rows(name):
    out = []
    for line in open(os.path.join(HERE, "golden", name)):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append([c.strip() for c in line.split("|")])
    return out


CASES = _rows("cache_bytes.txt")


@pytest.mark.parametrize("row", CASES, ids=[r[0] for r in CASES])
def test_printed_cache_sizes(row):
    name, L, hkv, d, n, B, p, printed, unit, cite = row
    got = formula.kv_cache_bytes(int(L), int(hkv), int(d), int(n), int(B), int(p))
    if unit == "B":
        assert got == int(printed)
    else:
        decimals = len(printed.split(".")[1]) if "." in printed else 0
        assert round(got / UNITS[unit], decimals) == float(printed), (got, cite)


RATIOS = _rows("cache_ratios.txt")


@pytest.mark.parametrize("row", RATIOS, ids=[r[0] for r in RATIOS])
def test_printed_savings_factors(row):
    name, H, Hkv, factor, cite = row
    mha = formula.kv_cache_bytes(32, int(H), 128, 1024, 1, 2)
    gqa = formula.kv_cache_bytes(32, int(Hkv), 128, 1024, 1, 2)
    assert mha == int(factor) * gqa


def test_per_token_is_cache_over_tokens():
    """The lesson record's per-token growth 2*L*Hkv*Dh*s is the payload
    estimate at T = 1, B = 1; the payload is linear in T and B."""
    assert formula.kv_bytes_per_token(80, 8, 128, 2) == 327680
    assert formula.kv_cache_bytes(80, 8, 128, 4096, 3, 2) == 3 * 4096 * 327680


def test_fractional_precision():
    """p = 0.5 for int4 ("10.3", section 2 list of p values)."""
    assert formula.kv_cache_bytes(80, 8, 128, 1, 1, 0.5) == 81920
    assert formula.kv_cache_bytes(80, 8, 128, 1, 1, 1) * 2 == 327680


def test_mqa_and_mla_forms():
    """MQA is the formula at one KV head ("10.3", 4.1); MLA stores one latent,
    no factor two ("10.3", 4.3)."""
    assert formula.kv_cache_bytes(80, 1, 128, 4096, 1, 2) * 64 == 10737418240
    assert formula.mla_cache_bytes(80, 512, 4096, 1, 2) == 80 * 512 * 4096 * 2
