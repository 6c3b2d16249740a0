"""The C ABI library loads and exports every function include/kvc.h
declares; host-only functions work without a GPU."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(kvc_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_decode_step():
    names = _declared()
    for must in ("kvc_alloc", "kvc_append", "kvc_decode_attn", "kvc_free", "kvc_get_error",
                 "kvc_cache_bytes", "kvc_workspace_bytes"):
        assert must in names


def test_every_declared_symbol_is_exported(kvc_library_path):
    out = subprocess.run(["nm", "-D", "--defined-only", kvc_library_path], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvc_\w+)$", out, flags=re.M))
    declared = set(_declared())
    assert declared <= exported, f"missing: {sorted(declared - exported)}"
    assert exported <= declared, f"exported but not declared: {sorted(exported - declared)}"


def test_binding_loads_and_host_functions(kvc_library_path):
    from static_kv_cache_gb300 import kvc
    assert kvc.kvc_abi_version() == 1
    assert kvc.kvc_status_str(0) == "ok"
    assert "unknown" in kvc.kvc_status_str(99)
    cfg = kvc.make_config(80, 1, 64, 64, 128, 4096, "fp16")
    assert kvc.kvc_cache_bytes(cfg) == 10737418240        # "10.3", section 2.1
    assert kvc.kvc_bytes_per_token(cfg) == 2621440         # "10.3", section 2.2
    assert kvc.kvc_check_config(cfg) == kvc.KVC_OK
    assert kvc.kvc_workspace_bytes(cfg) > 0


def test_product_formula_matches_the_printed_sizes(kvc_library_path):
    """The library's own size formula against every exact figure of the
    golden file (the oracle's formula is pinned to the same file)."""
    from static_kv_cache_gb300 import kvc
    from tests.test_oracle_formula import CASES, UNITS
    dt = {2: "bf16", 4: "fp32"}
    for name, L, hkv, d, n, B, p, printed, unit, cite in CASES:
        cfg = kvc.make_config(int(L), int(B), int(hkv), int(hkv), int(d), int(n), dt[int(p)])
        got = kvc.kvc_cache_bytes(cfg)
        if unit == "B":
            assert got == int(printed)
        else:
            decimals = len(printed.split(".")[1]) if "." in printed else 0
            assert round(got / UNITS[unit], decimals) == float(printed), name


@pytest.mark.parametrize("bad", [
    (0, 1, 8, 8, 128, 64, "bf16"), (1, 1, 8, 3, 128, 64, "bf16"), (1, 1, 8, 8, 0, 64, "bf16"),
    (1, 1, 8, 8, 128, 0, "bf16"), (1, 1, 8, 8, 128, 64, 9)])
def test_invalid_configs(kvc_library_path, bad):
    from static_kv_cache_gb300 import kvc
    cfg = kvc.make_config(*bad)
    assert kvc.kvc_check_config(cfg) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_cache_bytes(cfg) == 0
    assert kvc.kvc_workspace_bytes(cfg) == 0
    assert kvc.kvc_alloc(cfg, 16, 16, 16, 1 << 20)[0] == kvc.KVC_ERR_INVALID


@pytest.mark.parametrize("cfg", [(1, 1, 12, 1, 128, 64, "bf16"), (1, 1, 8, 8, 96, 64, "bf16"),
                                 (1, 1, 32, 1, 128, 64, "fp32"), (1, 1, 16, 1, 256, 64, "bf16"),
                                 (1, 1, 128, 1, 128, 64, "bf16")])
def test_unsupported_configs(kvc_library_path, cfg):
    from static_kv_cache_gb300 import kvc
    assert kvc.kvc_check_config(kvc.make_config(*cfg)) == kvc.KVC_ERR_UNSUPPORTED


@pytest.mark.parametrize("cfg", [(1, 1, 16, 1, 128, 64, "bf16"), (1, 1, 32, 1, 128, 64, "fp16"),
                                 (1, 1, 64, 1, 64, 64, "bf16"), (1, 1, 32, 2, 128, 64, "bf16")])
def test_multi_query_configs_are_supported(kvc_library_path, cfg):
    """Groups of 16, 32 and 64 query heads per KV head ("10.3", section 4.1)
    on 16-bit caches with d_h 64 or 128."""
    from static_kv_cache_gb300 import kvc
    assert kvc.kvc_check_config(kvc.make_config(*cfg)) == kvc.KVC_OK


def test_handle_calls_reject_null(kvc_library_path):
    from static_kv_cache_gb300 import kvc
    assert kvc.kvc_append(None, 0, 16, 16, 16, 1) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_decode_attn(None, 0, 16, 16, 0, 16) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_get_error(None) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_set_num_splits(None, 1) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_set_wait_timeout_ns(None, 1000) == kvc.KVC_ERR_INVALID
    kvc.kvc_free(None)


def test_all_configs_of_the_workloads_are_supported(kvc_library_path):
    from static_kv_cache_gb300 import kvc, synth
    for w in synth.WORKLOADS.values():
        if w.d_latent:
            continue   # MLA caches: test_mla_host_config
        cfg = kvc.make_config(w.n_layers, w.batch, w.n_heads, w.n_kv_heads, w.d_head, w.max_context, w.dtype)
        assert kvc.kvc_check_config(cfg) == kvc.KVC_OK, w.name


def test_mla_host_config(kvc_library_path):
    """The MLA cache size is the pages' one-tensor formula ("10.3", 4.3:
    n_layers * d_c * n_ctx * B * p), equal to the oracle's; unsupported and
    invalid shapes are refused on the host before any CUDA call."""
    import oracle
    from static_kv_cache_gb300 import kvc, synth
    w = synth.WORKLOADS["mla_dsv2"]
    cfg = kvc.make_mla_config(w.n_layers, w.batch, w.n_heads, w.d_head, w.d_latent, w.max_context, w.dtype)
    assert kvc.kvc_mla_cache_bytes(cfg) == oracle.mla_cache_bytes(w.n_layers, w.d_latent, w.max_context, w.batch, 2)
    assert kvc.kvc_mla_workspace_bytes(cfg) > 0
    assert kvc.kvc_mla_alloc(kvc.make_mla_config(1, 2, 16, 128, 96, 64, "bf16"), 16, 256, 1 << 30)[0] \
        == kvc.KVC_ERR_UNSUPPORTED
    assert kvc.kvc_mla_alloc(kvc.make_mla_config(1, 0, 16, 128, 512, 64, "bf16"), 16, 256, 1 << 30)[0] \
        == kvc.KVC_ERR_INVALID
    assert kvc.kvc_mla_cache_bytes(kvc.make_mla_config(1, 2, 16, 128, 512, 0, "bf16")) == 0
    assert kvc.kvc_mla_decode_attn(None, 0, 16, 16, 16, 16, 0, 16) == kvc.KVC_ERR_INVALID
    assert kvc.kvc_mla_get_error(None) == kvc.KVC_ERR_INVALID
    kvc.kvc_mla_free(None)
