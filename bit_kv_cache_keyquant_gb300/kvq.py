"""Thin Python binding of libkvq (include/kvq.h): argument marshalling only.

Every function has the name of its C entry point and takes torch tensors
(device memory) or plain integers; every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if libkvq.so is missing or
fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

_LIB_PATH = _build.LIB

KVQ_OK, KVQ_ERR_INVALID_ARG, KVQ_ERR_UNSUPPORTED, KVQ_ERR_MISALIGNED, KVQ_ERR_CUDA, KVQ_ERR_WORKSPACE = range(6)
KVQ_VARIANT_KIVI, KVQ_VARIANT_KITTY, KVQ_VARIANT_INT8, KVQ_VARIANT_INT8_TOKEN, KVQ_VARIANT_KIVI_PAGED = 0, 1, 2, 3, 4
KVQ_DEVICE_ERR_WAIT_TIMEOUT = 1
KVQ_DEVICE_ERR_CAPACITY = 2
KVQ_DEVICE_ERR_POOL = 4


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class kvq_config(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("bits_k", ctypes.c_int32), ("bits_v", ctypes.c_int32), ("group_k", ctypes.c_int32),
                ("group_v", ctypes.c_int32), ("residual", ctypes.c_int32), ("sink", ctypes.c_int32),
                ("boost_k", ctypes.c_int32), ("int8_block", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("int8_group", ctypes.c_int32)]


_P = ctypes.c_void_p


class kvq_kivi_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("seq_len", _P),
                ("k_codes", _P), ("k_sz", _P), ("v_codes", _P), ("v_sz", _P), ("k_res", _P), ("v_res", _P)]


class kvq_kivi_paged_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("seq_len", _P), ("page_table", _P),
                ("n_pages", ctypes.c_int32), ("pages", _P), ("k_res", _P), ("v_res", _P)]


class kvq_kitty_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("seq_len", _P),
                ("k_pages", _P), ("v_pages", _P), ("k_sink", _P), ("v_sink", _P), ("k_qbuf", _P),
                ("v_qbuf", _P), ("v_local", _P), ("page_table", _P),
                ("n_pages", ctypes.c_int32)]


class kvq_slot_pool(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int32), ("slots", _P), ("top", _P)]


class kvq_int8_token_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("seq_len", _P), ("slot_table", _P),
                ("n_slots", ctypes.c_int32), ("layer", ctypes.c_int32), ("seed", ctypes.c_uint64),
                ("k_codes", _P), ("v_codes", _P), ("k_scale", _P), ("v_scale", _P)]


class kvq_int8_cache(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_seq_len", ctypes.c_int32), ("seq_len", _P), ("req_id", _P),
                ("layer", ctypes.c_int32), ("seed", ctypes.c_uint64), ("k_codes", _P), ("v_codes", _P),
                ("k_scale", _P), ("v_scale", _P), ("k_tail", _P), ("v_tail", _P)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libkvq.so not built ({_LIB_PATH}); run __graft_entry__.build() or "
                          f"python -m bit_kv_cache_keyquant_gb300.build")
    lib = ctypes.CDLL(_LIB_PATH)
    S = ctypes.c_int
    i64, i32, sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    cfgp = ctypes.POINTER(kvq_config)
    sigs = {
        "kv_quant_key": (S, [cfgp, _P, i64, _P, _P, _P]),
        "kv_quant_value": (S, [cfgp, _P, i64, _P, _P, _P]),
        "kv_append_kivi": (S, [cfgp, ctypes.POINTER(kvq_kivi_cache), _P, _P, _P]),
        "kv_append_int8": (S, [cfgp, ctypes.POINTER(kvq_int8_cache), _P, _P, _P]),
        "kv_append_kitty": (S, [cfgp, ctypes.POINTER(kvq_kitty_cache), _P, _P, i32, _P]),
        "kvq_kivi_page_bytes": (sz, [cfgp]),
        "kv_quant_key_paged": (S, [cfgp, ctypes.POINTER(kvq_kivi_paged_cache), _P, i64, i32, i32, i32, _P]),
        "kv_quant_value_paged": (S, [cfgp, ctypes.POINTER(kvq_kivi_paged_cache), _P, i64, i32, i32, i32, _P]),
        "kv_append_kivi_paged": (S, [cfgp, ctypes.POINTER(kvq_kivi_paged_cache), ctypes.POINTER(kvq_slot_pool), _P,
                                     _P, _P]),
        "kv_release_kivi_paged": (S, [ctypes.POINTER(kvq_kivi_paged_cache), i32, ctypes.POINTER(kvq_slot_pool), _P]),
        "kv_decode_attn_kivi_paged": (S, [cfgp, ctypes.POINTER(kvq_kivi_paged_cache), _P, _P, _P, sz, _P]),
        "kv_quant_key_kitty_paged": (S, [cfgp, ctypes.POINTER(kvq_kitty_cache), _P, i64, i32, i32, i32, i32, _P]),
        "kv_quant_value_kitty_paged": (S, [cfgp, ctypes.POINTER(kvq_kitty_cache), _P, i64, i32, i32, i32, _P]),
        "kv_append_kitty_paged": (S, [cfgp, ctypes.POINTER(kvq_kitty_cache), ctypes.POINTER(kvq_slot_pool), _P, _P,
                                      i32, _P]),
        "kv_release_kitty": (S, [cfgp, ctypes.POINTER(kvq_kitty_cache), i32, ctypes.POINTER(kvq_slot_pool), _P]),
        "kv_quant_int8_token": (S, [cfgp, ctypes.POINTER(kvq_int8_token_cache), _P, i64, _P, i32, _P]),
        "kv_slot_pool_init": (S, [ctypes.POINTER(kvq_slot_pool), _P]),
        "kv_append_int8_token": (S, [cfgp, ctypes.POINTER(kvq_int8_token_cache), ctypes.POINTER(kvq_slot_pool), _P,
                                     _P, _P]),
        "kv_release_int8_token": (S, [ctypes.POINTER(kvq_int8_token_cache), i32, ctypes.POINTER(kvq_slot_pool), _P]),
        "kv_decode_attn_int8_token": (S, [cfgp, ctypes.POINTER(kvq_int8_token_cache), _P, _P, _P, sz, _P]),
        "kv_quant_key_kitty": (S, [cfgp, _P, i64, i32, _P, _P]),
        "kv_quant_value_kitty": (S, [cfgp, _P, i64, _P, _P]),
        "kv_quant_int8_dither": (S, [cfgp, _P, i64, _P, _P, _P, i32, i32, ctypes.c_uint64, _P, _P, _P]),
        "kvq_kitty_key_page_bytes": (sz, [cfgp]),
        "kvq_kitty_value_page_bytes": (sz, [cfgp]),
        "kv_decode_attn_plan": (S, [cfgp, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(sz)]),
        "kv_decode_attn": (S, [cfgp, ctypes.POINTER(kvq_kivi_cache), _P, _P, _P, sz, _P]),
        "kv_decode_attn_kitty": (S, [cfgp, ctypes.POINTER(kvq_kitty_cache), _P, _P, _P, sz, _P]),
        "kv_decode_attn_int8": (S, [cfgp, ctypes.POINTER(kvq_int8_cache), _P, _P, _P, sz, _P]),
        "kv_decode_attn_noalloc": (S, [cfgp, ctypes.POINTER(kvq_kivi_cache), _P, _P, _P]),
        "kv_decode_attn_stage1": (S, [cfgp, i32, _P, _P, _P, sz, _P]),
        "kv_decode_attn_merge": (S, [cfgp, i32, i32, i32, _P, sz, _P, _P]),
        "kvq_philox4x32_10": (S, [_P, _P, i64, _P, _P]),
        "kvq_get_device_error": (S, [ctypes.POINTER(ctypes.c_uint32)]),
        "kvq_status_string": (ctypes.c_char_p, [S]),
        "kvq_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()

EXPORTED = ("kv_quant_key", "kv_quant_value", "kv_append_kivi", "kv_append_int8", "kv_append_kitty",
            "kv_quant_key_kitty", "kv_quant_value_kitty", "kv_quant_int8_dither", "kv_quant_int8_token",
            "kv_slot_pool_init", "kv_append_int8_token", "kv_release_int8_token", "kvq_kivi_page_bytes",
            "kv_quant_key_paged", "kv_quant_value_paged", "kv_append_kivi_paged", "kv_release_kivi_paged",
            "kv_decode_attn_kivi_paged", "kv_quant_key_kitty_paged", "kv_quant_value_kitty_paged",
            "kv_append_kitty_paged", "kv_release_kitty",
            "kvq_kitty_key_page_bytes", "kvq_kitty_value_page_bytes", "kv_decode_attn_plan", "kv_decode_attn",
            "kv_decode_attn_kitty", "kv_decode_attn_int8", "kv_decode_attn_int8_token", "kv_decode_attn_noalloc",
            "kv_decode_attn_stage1", "kv_decode_attn_merge",
            "kvq_philox4x32_10", "kvq_get_device_error", "kvq_status_string", "kvq_version")


def library_path() -> str:
    return _LIB_PATH


def status_string(s: int) -> str:
    return _lib.kvq_status_string(s).decode()


def version() -> str:
    return _lib.kvq_version().decode()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != KVQ_OK:
        raise KvqError(status, what)


def make_config(head_dim=128, n_q_heads=32, n_kv_heads=32, bits_k=2, bits_v=2, group_k=32, group_v=32,
                residual=128, sink=32, boost_k=16, int8_block=256, sm_scale=0.0, int8_group=32) -> kvq_config:
    return kvq_config(head_dim, n_q_heads, n_kv_heads, bits_k, bits_v, group_k, group_v, residual, sink, boost_k,
                      int8_block, sm_scale, int8_group)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def kv_quant_key(cfg, k, n_groups, codes, sz, stream=None):
    _check(_lib.kv_quant_key(ctypes.byref(cfg), _ptr(k), n_groups, _ptr(codes), _ptr(sz), _stream(stream)),
           "kv_quant_key")


def kv_quant_value(cfg, v, n_tokens, codes, sz, stream=None):
    _check(_lib.kv_quant_value(ctypes.byref(cfg), _ptr(v), n_tokens, _ptr(codes), _ptr(sz), _stream(stream)),
           "kv_quant_value")


def kv_append_kivi(cfg, cache, k_new, v_new, stream=None):
    """Append one token per (batch row, kv head): k_new, v_new fp16 [B][Hkv][D]."""
    _check(_lib.kv_append_kivi(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k_new), _ptr(v_new), _stream(stream)),
           "kv_append_kivi")


def kv_append_int8(cfg, cache, k_new, v_new, stream=None):
    """Append one token per (batch row, kv head) to an INT8 cache: k_new, v_new fp16 [B][Hkv][D]."""
    _check(_lib.kv_append_int8(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k_new), _ptr(v_new), _stream(stream)),
           "kv_append_int8")


def kv_append_kitty(cfg, cache, k_new, v_new, score_mode=0, stream=None):
    """Append one token per (batch row, kv head) to a Kitty cache: k_new, v_new fp16 [B][Hkv][D]."""
    _check(_lib.kv_append_kitty(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k_new), _ptr(v_new), score_mode,
                                _stream(stream)), "kv_append_kitty")


def kvq_kivi_page_bytes(cfg) -> int:
    return int(_lib.kvq_kivi_page_bytes(ctypes.byref(cfg)))


def kv_quant_key_paged(cfg, cache, k, n_groups, group0, row, kv_head, stream=None):
    _check(_lib.kv_quant_key_paged(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k), n_groups, group0, row, kv_head,
                                   _stream(stream)), "kv_quant_key_paged")


def kv_quant_value_paged(cfg, cache, v, n_tokens, tok0, row, kv_head, stream=None):
    _check(_lib.kv_quant_value_paged(ctypes.byref(cfg), ctypes.byref(cache), _ptr(v), n_tokens, tok0, row, kv_head,
                                     _stream(stream)), "kv_quant_value_paged")


def kv_append_kivi_paged(cfg, cache, pool, k_new, v_new, stream=None):
    _check(_lib.kv_append_kivi_paged(ctypes.byref(cfg), ctypes.byref(cache), ctypes.byref(pool), _ptr(k_new),
                                     _ptr(v_new), _stream(stream)), "kv_append_kivi_paged")


def kv_release_kivi_paged(cache, row, pool, stream=None):
    _check(_lib.kv_release_kivi_paged(ctypes.byref(cache), row, ctypes.byref(pool), _stream(stream)),
           "kv_release_kivi_paged")


def kv_decode_attn_kivi_paged(cfg, cache, q, out, workspace, workspace_bytes, stream=None):
    _check(_lib.kv_decode_attn_kivi_paged(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out),
                                          _ptr(workspace), workspace_bytes, _stream(stream)),
           "kv_decode_attn_kivi_paged")


def kv_quant_key_kitty_paged(cfg, cache, k, n_pages, page0, row, kv_head, score_mode=0, stream=None):
    _check(_lib.kv_quant_key_kitty_paged(ctypes.byref(cfg), ctypes.byref(cache), _ptr(k), n_pages, page0, row, kv_head,
                                         score_mode, _stream(stream)), "kv_quant_key_kitty_paged")


def kv_quant_value_kitty_paged(cfg, cache, v, n_pages, page0, row, kv_head, stream=None):
    _check(_lib.kv_quant_value_kitty_paged(ctypes.byref(cfg), ctypes.byref(cache), _ptr(v), n_pages, page0, row,
                                           kv_head, _stream(stream)), "kv_quant_value_kitty_paged")


def kv_append_kitty_paged(cfg, cache, pool, k_new, v_new, score_mode=0, stream=None):
    _check(_lib.kv_append_kitty_paged(ctypes.byref(cfg), ctypes.byref(cache), ctypes.byref(pool), _ptr(k_new),
                                      _ptr(v_new), score_mode, _stream(stream)), "kv_append_kitty_paged")


def kv_release_kitty(cfg, cache, row, pool, stream=None):
    _check(_lib.kv_release_kitty(ctypes.byref(cfg), ctypes.byref(cache), row, ctypes.byref(pool), _stream(stream)),
           "kv_release_kitty")


def kv_quant_int8_token(cfg, cache, x, n, slots, kv_sel, stream=None):
    """Quantize n tokens x fp16 [n][Hkv][D] into pool slots slots int32 [n] (keys: kv_sel 0, values: 1)."""
    _check(_lib.kv_quant_int8_token(ctypes.byref(cfg), ctypes.byref(cache), _ptr(x), n, _ptr(slots), kv_sel,
                                    _stream(stream)), "kv_quant_int8_token")


def kv_slot_pool_init(pool, stream=None):
    _check(_lib.kv_slot_pool_init(ctypes.byref(pool), _stream(stream)), "kv_slot_pool_init")


def kv_append_int8_token(cfg, cache, pool, k_new, v_new, stream=None):
    """Append one token per request (fp16 [B][Hkv][D]) into slots taken from the pool."""
    _check(_lib.kv_append_int8_token(ctypes.byref(cfg), ctypes.byref(cache), ctypes.byref(pool), _ptr(k_new),
                                     _ptr(v_new), _stream(stream)), "kv_append_int8_token")


def kv_release_int8_token(cache, row, pool, stream=None):
    _check(_lib.kv_release_int8_token(ctypes.byref(cache), row, ctypes.byref(pool), _stream(stream)),
           "kv_release_int8_token")


def kv_quant_key_kitty(cfg, k, n_pages, score_mode, pages, stream=None):
    _check(_lib.kv_quant_key_kitty(ctypes.byref(cfg), _ptr(k), n_pages, score_mode, _ptr(pages), _stream(stream)),
           "kv_quant_key_kitty")


def kv_quant_value_kitty(cfg, v, n_pages, pages, stream=None):
    _check(_lib.kv_quant_value_kitty(ctypes.byref(cfg), _ptr(v), n_pages, _ptr(pages), _stream(stream)),
           "kv_quant_value_kitty")


def kv_quant_int8_dither(cfg, x, n_blocks, req_id, kv_head, tok0, layer, kv_sel, seed, codes, scale, stream=None):
    _check(_lib.kv_quant_int8_dither(ctypes.byref(cfg), _ptr(x), n_blocks, _ptr(req_id), _ptr(kv_head), _ptr(tok0),
                                     layer, kv_sel, seed, _ptr(codes), _ptr(scale), _stream(stream)),
           "kv_quant_int8_dither")


def kvq_kitty_key_page_bytes(cfg) -> int:
    return _lib.kvq_kitty_key_page_bytes(ctypes.byref(cfg))


def kvq_kitty_value_page_bytes(cfg) -> int:
    return _lib.kvq_kitty_value_page_bytes(ctypes.byref(cfg))


def kv_decode_attn_plan(cfg, variant, batch, max_seq_len):
    n = ctypes.c_int32()
    b = ctypes.c_size_t()
    _check(_lib.kv_decode_attn_plan(ctypes.byref(cfg), variant, batch, max_seq_len, ctypes.byref(n), ctypes.byref(b)),
           "kv_decode_attn_plan")
    return n.value, b.value


def kv_decode_attn(cfg, cache, q, out, workspace, workspace_bytes, stream=None):
    _check(_lib.kv_decode_attn(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out), _ptr(workspace),
                               workspace_bytes, _stream(stream)), "kv_decode_attn")


def kv_decode_attn_kitty(cfg, cache, q, out, workspace, workspace_bytes, stream=None):
    _check(_lib.kv_decode_attn_kitty(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out), _ptr(workspace),
                                     workspace_bytes, _stream(stream)), "kv_decode_attn_kitty")


def kv_decode_attn_int8(cfg, cache, q, out, workspace, workspace_bytes, stream=None):
    _check(_lib.kv_decode_attn_int8(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out), _ptr(workspace),
                                    workspace_bytes, _stream(stream)), "kv_decode_attn_int8")


def kv_decode_attn_int8_token(cfg, cache, q, out, workspace, workspace_bytes, stream=None):
    _check(_lib.kv_decode_attn_int8_token(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out),
                                          _ptr(workspace), workspace_bytes, _stream(stream)),
           "kv_decode_attn_int8_token")


def kv_decode_attn_noalloc(cfg, cache, q, out, stream=None):
    """kv_decode_attn without a caller workspace (fixed scratch inside the library)."""
    _check(_lib.kv_decode_attn_noalloc(ctypes.byref(cfg), ctypes.byref(cache), _ptr(q), _ptr(out), _stream(stream)),
           "kv_decode_attn_noalloc")


def kv_decode_attn_stage1(cfg, variant, cache, q, workspace, workspace_bytes, stream=None):
    _check(_lib.kv_decode_attn_stage1(ctypes.byref(cfg), variant, ctypes.byref(cache), _ptr(q), _ptr(workspace),
                                      workspace_bytes, _stream(stream)), "kv_decode_attn_stage1")


def kv_decode_attn_merge(cfg, variant, batch, max_seq_len, workspace, workspace_bytes, out, stream=None):
    _check(_lib.kv_decode_attn_merge(ctypes.byref(cfg), variant, batch, max_seq_len, _ptr(workspace),
                                     workspace_bytes, _ptr(out), _stream(stream)), "kv_decode_attn_merge")


def kvq_philox4x32_10(ctr, key, n, out, stream=None):
    _check(_lib.kvq_philox4x32_10(_ptr(ctr), _ptr(key), n, _ptr(out), _stream(stream)), "kvq_philox4x32_10")


def kvq_get_device_error() -> int:
    v = ctypes.c_uint32()
    _check(_lib.kvq_get_device_error(ctypes.byref(v)), "kvq_get_device_error")
    return v.value


def raw_call(name, *args):
    """Call a C entry point with raw ctypes arguments and return its status."""
    return getattr(_lib, name)(*args)
