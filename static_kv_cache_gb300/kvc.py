"""ctypes binding of libkvc.so -- argument marshalling only.

Every function here has the name and argument order of the C function in
``include/kvc.h`` and returns what it returns (a ``kvc_status`` int, a size,
or, for ``kvc_alloc``, ``(status, handle)``).  Pointer arguments accept an
int address or any object with ``data_ptr()`` (a torch tensor); stream
arguments accept an int handle, ``None`` (legacy default stream) or any object
with ``cuda_stream`` (a torch stream).  No computation happens in Python.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvc.so")

KVC_OK = 0
KVC_ERR_INVALID = 1
KVC_ERR_CAPACITY = 2
KVC_ERR_CUDA = 3
KVC_ERR_WORKSPACE = 4
KVC_ERR_TIMEOUT = 5
KVC_ERR_DEVICE_INDEX = 6
KVC_ERR_UNSUPPORTED = 7
KVC_ERR_ALIGNMENT = 8

KVC_BF16 = 0
KVC_FP32 = 1
KVC_FP16 = 2
KVC_INT8 = 3
DTYPE_CODES = {"bf16": KVC_BF16, "fp32": KVC_FP32, "fp16": KVC_FP16, "int8": KVC_INT8}

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
        "(the decode path has no fallback without its CUDA library)")

_lib = ctypes.CDLL(LIB_PATH)


class kvc_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("d_head", ctypes.c_int32), ("max_context", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class KvcError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__(f"{what}: {kvc_status_str(status)} ({status})" if what
                         else f"{kvc_status_str(status)} ({status})")
        self.status = status


_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_u64 = ctypes.c_uint64
_cfgp = ctypes.POINTER(kvc_config)

_lib.kvc_abi_version.restype = _i32
_lib.kvc_status_str.argtypes = [_i32]
_lib.kvc_status_str.restype = ctypes.c_char_p
_lib.kvc_check_config.argtypes = [_cfgp]
_lib.kvc_check_config.restype = _i32
for _n in ("kvc_cache_bytes", "kvc_bytes_per_token", "kvc_workspace_bytes", "kvc_scale_bytes"):
    getattr(_lib, _n).argtypes = [_cfgp]
    getattr(_lib, _n).restype = _u64
_lib.kvc_alloc.argtypes = [_cfgp, _vp, _vp, _vp, _u64, ctypes.POINTER(_vp)]
_lib.kvc_alloc.restype = _i32
_lib.kvc_alloc_scaled.argtypes = [_cfgp, _vp, _vp, _vp, _vp, _vp, _u64, ctypes.POINTER(_vp)]
_lib.kvc_alloc_scaled.restype = _i32
_lib.kvc_alloc_paged.argtypes = [_cfgp, _vp, _vp, _i32, _vp, _vp, _u64, ctypes.POINTER(_vp)]
_lib.kvc_alloc_paged.restype = _i32
_lib.kvc_pool_bytes.argtypes = [_cfgp, _i32]
_lib.kvc_pool_bytes.restype = _u64
_lib.kvc_free.argtypes = [_vp]
_lib.kvc_free.restype = None
_lib.kvc_set_num_splits.argtypes = [_vp, _i32]
_lib.kvc_set_num_splits.restype = _i32
_lib.kvc_append.argtypes = [_vp, _i32, _vp, _vp, _vp, _i32, _vp]
_lib.kvc_append.restype = _i32
_lib.kvc_decode_attn.argtypes = [_vp, _i32, _vp, _vp, _i32, _vp, _vp]
_lib.kvc_decode_attn.restype = _i32
_lib.kvc_decode_step.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp]
_lib.kvc_decode_step.restype = _i32
_lib.kvc_prefill_attn.argtypes = [_vp, _i32, _vp, _vp, _i32, _vp, _vp]
_lib.kvc_prefill_attn.restype = _i32
_lib.kvc_decode_attn_static.argtypes = [_cfgp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp]
_lib.kvc_decode_attn_static.restype = _i32
_lib.kvc_get_error.argtypes = [_vp, _vp]
_lib.kvc_get_error.restype = _i32
_lib.kvc_static_get_error.argtypes = [_vp]
_lib.kvc_static_get_error.restype = _i32
_lib.kvc_set_wait_timeout_ns.argtypes = [_vp, _u64]
_lib.kvc_set_wait_timeout_ns.restype = _i32


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def make_config(n_layers, batch, n_heads, n_kv_heads, d_head, max_context, dtype) -> kvc_config:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return kvc_config(n_layers, batch, n_heads, n_kv_heads, d_head, max_context, code)


def kvc_abi_version() -> int:
    return _lib.kvc_abi_version()


def kvc_status_str(status: int) -> str:
    return _lib.kvc_status_str(int(status)).decode()


def kvc_check_config(cfg: kvc_config) -> int:
    return _lib.kvc_check_config(ctypes.byref(cfg))


def kvc_cache_bytes(cfg: kvc_config) -> int:
    return _lib.kvc_cache_bytes(ctypes.byref(cfg))


def kvc_bytes_per_token(cfg: kvc_config) -> int:
    return _lib.kvc_bytes_per_token(ctypes.byref(cfg))


def kvc_workspace_bytes(cfg: kvc_config) -> int:
    return _lib.kvc_workspace_bytes(ctypes.byref(cfg))


def kvc_alloc(cfg: kvc_config, k_base, v_base, workspace, ws_bytes: int):
    h = _vp()
    st = _lib.kvc_alloc(ctypes.byref(cfg), _ptr(k_base), _ptr(v_base), _ptr(workspace),
                        int(ws_bytes), ctypes.byref(h))
    return st, (h.value if st == KVC_OK else None)


def kvc_scale_bytes(cfg: kvc_config) -> int:
    return _lib.kvc_scale_bytes(ctypes.byref(cfg))


def kvc_alloc_scaled(cfg: kvc_config, k_base, v_base, k_scale, v_scale, workspace, ws_bytes: int):
    h = _vp()
    st = _lib.kvc_alloc_scaled(ctypes.byref(cfg), _ptr(k_base), _ptr(v_base), _ptr(k_scale), _ptr(v_scale),
                               _ptr(workspace), int(ws_bytes), ctypes.byref(h))
    return st, (h.value if st == KVC_OK else None)


def kvc_pool_bytes(cfg: kvc_config, num_blocks: int) -> int:
    return _lib.kvc_pool_bytes(ctypes.byref(cfg), int(num_blocks))


def kvc_alloc_paged(cfg: kvc_config, k_pool, v_pool, num_blocks: int, block_table, workspace, ws_bytes: int):
    h = _vp()
    st = _lib.kvc_alloc_paged(ctypes.byref(cfg), _ptr(k_pool), _ptr(v_pool), int(num_blocks), _ptr(block_table),
                              _ptr(workspace), int(ws_bytes), ctypes.byref(h))
    return st, (h.value if st == KVC_OK else None)


def kvc_free(h) -> None:
    _lib.kvc_free(h)


def kvc_set_num_splits(h, n: int) -> int:
    return _lib.kvc_set_num_splits(h, int(n))


def kvc_set_wait_timeout_ns(h, ns: int) -> int:
    return _lib.kvc_set_wait_timeout_ns(h, int(ns))


def kvc_append(h, layer: int, k_new, v_new, cache_index, T_new: int, stream=None) -> int:
    return _lib.kvc_append(h, int(layer), _ptr(k_new), _ptr(v_new), _ptr(cache_index),
                           int(T_new), _stream(stream))


def kvc_decode_attn(h, layer: int, q, valid_len, max_valid_hint: int, out, stream=None) -> int:
    return _lib.kvc_decode_attn(h, int(layer), _ptr(q), _ptr(valid_len), int(max_valid_hint),
                                _ptr(out), _stream(stream))


def kvc_decode_step(h, layer: int, q, k_new, v_new, valid_len, max_valid_hint: int, out, stream=None) -> int:
    return _lib.kvc_decode_step(h, int(layer), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(valid_len),
                                int(max_valid_hint), _ptr(out), _stream(stream))


def kvc_prefill_attn(h, layer: int, q, cache_index, T_new: int, out, stream=None) -> int:
    return _lib.kvc_prefill_attn(h, int(layer), _ptr(q), _ptr(cache_index), int(T_new), _ptr(out),
                                 _stream(stream))


def kvc_decode_attn_static(cfg: kvc_config, layer: int, k_base, v_base, q, valid_len,
                           max_valid_hint: int, out, stream=None) -> int:
    return _lib.kvc_decode_attn_static(ctypes.byref(cfg), int(layer), _ptr(k_base), _ptr(v_base),
                                       _ptr(q), _ptr(valid_len), int(max_valid_hint), _ptr(out),
                                       _stream(stream))


def kvc_get_error(h, stream=None) -> int:
    return _lib.kvc_get_error(h, _stream(stream))


def kvc_static_get_error(stream=None) -> int:
    return _lib.kvc_static_get_error(_stream(stream))


def check(status: int, what: str = "") -> None:
    """Raise KvcError unless status is KVC_OK."""
    if status != KVC_OK:
        raise KvcError(status, what)


# ---- MLA latent cache
class kvc_mla_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("d_head", ctypes.c_int32),
                ("d_latent", ctypes.c_int32), ("max_context", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_mcfgp = ctypes.POINTER(kvc_mla_config)
for _n in ("kvc_mla_cache_bytes", "kvc_mla_workspace_bytes"):
    getattr(_lib, _n).argtypes = [_mcfgp]
    getattr(_lib, _n).restype = _u64
_lib.kvc_mla_alloc.argtypes = [_mcfgp, _vp, _vp, _u64, ctypes.POINTER(_vp)]
_lib.kvc_mla_alloc.restype = _i32
_lib.kvc_mla_free.argtypes = [_vp]
_lib.kvc_mla_free.restype = None
_lib.kvc_mla_set_num_splits.argtypes = [_vp, _i32]
_lib.kvc_mla_set_num_splits.restype = _i32
_lib.kvc_mla_append.argtypes = [_vp, _i32, _vp, _vp, _i32, _vp]
_lib.kvc_mla_append.restype = _i32
_lib.kvc_mla_decode_attn.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, _vp]
_lib.kvc_mla_decode_attn.restype = _i32
_lib.kvc_mla_decode_step.argtypes = [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp]
_lib.kvc_mla_decode_step.restype = _i32
_lib.kvc_mla_get_error.argtypes = [_vp, _vp]
_lib.kvc_mla_get_error.restype = _i32


def make_mla_config(n_layers, batch, n_heads, d_head, d_latent, max_context, dtype) -> kvc_mla_config:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return kvc_mla_config(n_layers, batch, n_heads, d_head, d_latent, max_context, code)


def kvc_mla_cache_bytes(cfg: kvc_mla_config) -> int:
    return _lib.kvc_mla_cache_bytes(ctypes.byref(cfg))


def kvc_mla_workspace_bytes(cfg: kvc_mla_config) -> int:
    return _lib.kvc_mla_workspace_bytes(ctypes.byref(cfg))


def kvc_mla_alloc(cfg: kvc_mla_config, c_base, workspace, ws_bytes: int):
    h = _vp()
    st = _lib.kvc_mla_alloc(ctypes.byref(cfg), _ptr(c_base), _ptr(workspace), int(ws_bytes), ctypes.byref(h))
    return st, (h.value if st == KVC_OK else None)


def kvc_mla_free(h) -> None:
    _lib.kvc_mla_free(h)


def kvc_mla_set_num_splits(h, n: int) -> int:
    return _lib.kvc_mla_set_num_splits(h, int(n))


def kvc_mla_append(h, layer: int, c_new, cache_index, T_new: int, stream=None) -> int:
    return _lib.kvc_mla_append(h, int(layer), _ptr(c_new), _ptr(cache_index), int(T_new), _stream(stream))


def kvc_mla_decode_attn(h, layer: int, q, w_uk, w_uv, valid_len, max_valid_hint: int, out, stream=None) -> int:
    return _lib.kvc_mla_decode_attn(h, int(layer), _ptr(q), _ptr(w_uk), _ptr(w_uv), _ptr(valid_len),
                                    int(max_valid_hint), _ptr(out), _stream(stream))


def kvc_mla_decode_step(h, layer: int, q, c_new, w_uk, w_uv, valid_len, max_valid_hint: int, out,
                        stream=None) -> int:
    return _lib.kvc_mla_decode_step(h, int(layer), _ptr(q), _ptr(c_new), _ptr(w_uk), _ptr(w_uv),
                                    _ptr(valid_len), int(max_valid_hint), _ptr(out), _stream(stream))


def kvc_mla_get_error(h, stream=None) -> int:
    return _lib.kvc_mla_get_error(h, _stream(stream))
