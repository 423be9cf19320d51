"""CPU checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def K():
    from bit_kv_cache_keyquant_gb300 import build
    build.build()
    from bit_kv_cache_keyquant_gb300 import kvq
    return kvq


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:KVQ_API\s+)?(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n.startswith(("kv_", "kvq_"))))


def test_header_symbols_exported(K):
    names = declared_functions()
    assert len(names) >= 17
    lib = ctypes.CDLL(K.library_path())
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(K.EXPORTED) == names


def test_oracle_and_library_share_no_code():
    """Neither side imports or includes the other (inputs.py holds no method arithmetic)."""
    pkg = os.path.join(ROOT, "bit_kv_cache_keyquant_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            src = open(os.path.join(dirpath, f), errors="ignore").read() if f.endswith((".py", ".cu", ".cuh", ".h")) else ""
            assert not re.search(r"^\s*(from\s+oracle|import\s+oracle)", src, flags=re.M), f
            assert not re.search(r'#include\s+[<"].*oracle', src), f
    for f in ("oracle.py", "kvq_oracle.c"):
        src = open(os.path.join(ROOT, "oracle", f)).read()
        assert not re.search(r"^\s*(from|import)\s+bit_kv_cache_keyquant_gb300", src, flags=re.M), f
        assert "#include \"../" not in src and "kvq.h" not in src.replace("kvq.h)", ""), f


def test_status_strings(K):
    assert K.status_string(0) == "ok"
    assert "aligned" in K.status_string(3)
    assert K.version().startswith("kvq")


def _call_quant_key(K, cfg, k=16, codes=16, sz=16, n=1):
    return K.raw_call("kv_quant_key", ctypes.byref(cfg), k, n, codes, sz, None)


def test_validation_without_gpu(K):
    good = K.make_config()
    bad_d = K.make_config(head_dim=64)
    assert _call_quant_key(K, bad_d) == K.KVQ_ERR_UNSUPPORTED
    assert _call_quant_key(K, K.make_config(bits_k=3)) == K.KVQ_ERR_UNSUPPORTED
    assert _call_quant_key(K, K.make_config(bits_k=8)) == K.KVQ_ERR_UNSUPPORTED
    assert _call_quant_key(K, K.make_config(bits_k=4), k=None) == K.KVQ_ERR_INVALID_ARG   # 4 bits is accepted
    assert _call_quant_key(K, K.make_config(residual=100)) == K.KVQ_ERR_UNSUPPORTED     # R % G != 0
    assert _call_quant_key(K, K.make_config(n_q_heads=30, n_kv_heads=8)) == K.KVQ_ERR_INVALID_ARG
    assert _call_quant_key(K, good, k=None) == K.KVQ_ERR_INVALID_ARG
    assert _call_quant_key(K, good, codes=0x1001) == K.KVQ_ERR_MISALIGNED
    assert _call_quant_key(K, good, n=-1) == K.KVQ_ERR_INVALID_ARG
    assert _call_quant_key(K, good, k=None, n=0) == K.KVQ_OK        # nothing to do, nothing launched
    assert K.raw_call("kv_quant_key", None, 16, 1, 16, 16, None) == K.KVQ_ERR_INVALID_ARG
    kitty = K.make_config(group_k=128, n_q_heads=32, n_kv_heads=8)
    assert K.kvq_kitty_key_page_bytes(kitty) == 5248
    assert K.kvq_kitty_value_page_bytes(kitty) == 4608
    assert K.raw_call("kv_quant_key_kitty", ctypes.byref(kitty), 16, 1, 2, 16, None) == K.KVQ_ERR_INVALID_ARG
    cache = K.kvq_kivi_cache(2, 512, 16, 16, 16, 16, 16, 16, 16)
    assert K.raw_call("kv_append_kivi", ctypes.byref(good), ctypes.byref(cache), None, 16, None) == K.KVQ_ERR_INVALID_ARG
    assert K.raw_call("kv_append_kivi", ctypes.byref(good), ctypes.byref(cache), 16, 0x1004, None) == \
        K.KVQ_ERR_MISALIGNED
    assert K.raw_call("kv_append_kivi", ctypes.byref(good), None, 16, 16, None) == K.KVQ_ERR_INVALID_ARG
    assert K.raw_call("kv_append_kivi", ctypes.byref(K.make_config(bits_v=1)), ctypes.byref(cache), 16, 16,
                      None) == K.KVQ_ERR_UNSUPPORTED
    kc = K.kvq_kitty_cache(2, 512, 16, 16, 16, 16, 16, 16, 16, 16)
    assert K.raw_call("kv_append_kitty", ctypes.byref(kitty), ctypes.byref(kc), 16, 16, 2, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert K.raw_call("kv_append_kitty", ctypes.byref(kitty), ctypes.byref(kc), 16, None, 0, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert K.raw_call("kv_append_kitty", ctypes.byref(kitty), ctypes.byref(kc), 0x1004, 16, 0, None) == \
        K.KVQ_ERR_MISALIGNED
    assert K.raw_call("kv_append_kitty", ctypes.byref(K.make_config(group_k=64)), ctypes.byref(kc), 16, 16, 0,
                      None) == K.KVQ_ERR_UNSUPPORTED
    i8 = K.make_config(int8_block=200)
    assert K.raw_call("kv_quant_int8_dither", ctypes.byref(i8), 16, 1, 16, 16, 16, 0, 0, 0, 16, 16,
                      None) == K.KVQ_ERR_UNSUPPORTED


def test_int8_token_validation_without_gpu(K):
    cfg = K.make_config(n_q_heads=64, n_kv_heads=8)
    c = K.kvq_int8_token_cache(4, 1024, 16, 16, 4096, 3, 7, 16, 16, 16, 16)
    pool = K.kvq_slot_pool(4096, 16, 16)
    call = K.raw_call
    assert call("kv_quant_int8_token", ctypes.byref(cfg), ctypes.byref(c), 16, 5, 16, 2, None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_quant_int8_token", ctypes.byref(cfg), ctypes.byref(c), 16, -1, 16, 0, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert call("kv_quant_int8_token", ctypes.byref(cfg), ctypes.byref(c), 0x1008, 5, 16, 0, None) == \
        K.KVQ_ERR_MISALIGNED
    assert call("kv_quant_int8_token", ctypes.byref(cfg), ctypes.byref(c), 16, 0, None, 0, None) == K.KVQ_OK
    assert call("kv_quant_int8_token", ctypes.byref(K.make_config(int8_group=48)), ctypes.byref(c), 16, 5, 16, 0,
                None) == K.KVQ_ERR_UNSUPPORTED
    assert call("kv_quant_int8_token", ctypes.byref(K.make_config(int8_group=0)), ctypes.byref(c), 16, 5, 16, 0,
                None) == K.KVQ_ERR_INVALID_ARG
    bad_layer = K.kvq_int8_token_cache(4, 1024, 16, 16, 4096, 1 << 15, 7, 16, 16, 16, 16)
    assert call("kv_append_int8_token", ctypes.byref(cfg), ctypes.byref(bad_layer), ctypes.byref(pool), 16, 16,
                None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_append_int8_token", ctypes.byref(cfg), ctypes.byref(c), ctypes.byref(K.kvq_slot_pool(0, 16, 16)),
                16, 16, None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_append_int8_token", ctypes.byref(cfg), ctypes.byref(c), None, 16, 16, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert call("kv_release_int8_token", ctypes.byref(c), 4, ctypes.byref(pool), None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_slot_pool_init", ctypes.byref(K.kvq_slot_pool(8, 16, 0x1004)), None) == K.KVQ_ERR_MISALIGNED
    wide = K.make_config(n_q_heads=72, n_kv_heads=8)                 # 9 query heads per kv head
    assert call("kv_decode_attn_int8_token", ctypes.byref(wide), ctypes.byref(c), 16, 16, 16, 1 << 30, None) == \
        K.KVQ_ERR_UNSUPPORTED
    n, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8_TOKEN, 4, 1024)
    assert call("kv_decode_attn_int8_token", ctypes.byref(cfg), ctypes.byref(c), 16, 16, 16, wsb - 1, None) == \
        K.KVQ_ERR_WORKSPACE


def test_kivi_paged_validation_without_gpu(K):
    cfg = K.make_config(n_q_heads=8, n_kv_heads=2)
    assert K.kvq_kivi_page_bytes(cfg) == 4096 + 2048 + 4096 + 2048
    assert K.kvq_kivi_page_bytes(K.make_config(bits_k=4, bits_v=4)) == 8192 + 2048 + 8192 + 2048
    c = K.kvq_kivi_paged_cache(2, 1000, 16, 16, 64, 16, 16, 16)
    call = K.raw_call
    assert call("kv_quant_key_paged", ctypes.byref(cfg), ctypes.byref(c), 16, 4, 0, 2, 0, None) == \
        K.KVQ_ERR_INVALID_ARG                                           # row out of range
    assert call("kv_quant_key_paged", ctypes.byref(cfg), ctypes.byref(c), 16, 4, 0, 0, 2, None) == \
        K.KVQ_ERR_INVALID_ARG                                           # kv head out of range
    assert call("kv_quant_key_paged", ctypes.byref(cfg), ctypes.byref(c), 16, 33, 0, 0, 0, None) == \
        K.KVQ_ERR_INVALID_ARG                                           # 33 groups of 32 > 1024 tokens
    assert call("kv_quant_value_paged", ctypes.byref(cfg), ctypes.byref(c), 16, 10, 1020, 0, 0, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert call("kv_quant_value_paged", ctypes.byref(cfg), ctypes.byref(c), 0x1002, 10, 0, 0, 0, None) == \
        K.KVQ_ERR_MISALIGNED
    assert call("kv_append_kivi_paged", ctypes.byref(cfg), ctypes.byref(c), None, 16, 16, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert call("kv_release_kivi_paged", ctypes.byref(c), -1, ctypes.byref(K.kvq_slot_pool(8, 16, 16)), None) == \
        K.KVQ_ERR_INVALID_ARG
    n, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI_PAGED, 2, 1000)
    assert call("kv_decode_attn_kivi_paged", ctypes.byref(cfg), ctypes.byref(c), 16, 16, 16, wsb - 1, None) == \
        K.KVQ_ERR_WORKSPACE
    assert call("kv_decode_attn_kivi_paged", ctypes.byref(K.make_config(bits_k=3)), ctypes.byref(c), 16, 16, 16, wsb,
                None) == K.KVQ_ERR_UNSUPPORTED


def test_kitty_paged_validation_without_gpu(K):
    cfg = K.make_config(n_q_heads=8, n_kv_heads=2, group_k=128)
    dense = K.kvq_kitty_cache(2, 1000, 16, 16, 16, 16, 16, 16, 16, 16)
    paged = K.kvq_kitty_cache(2, 1000, 16, 16, 16, 16, 16, 16, 16, 16, 16, 8)
    pool = K.kvq_slot_pool(8, 16, 16)
    call = K.raw_call
    assert call("kv_append_kitty", ctypes.byref(cfg), ctypes.byref(paged), 16, 16, 0, None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_append_kitty_paged", ctypes.byref(cfg), ctypes.byref(dense), ctypes.byref(pool), 16, 16, 0,
                None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_append_kitty_paged", ctypes.byref(cfg), ctypes.byref(paged), ctypes.byref(pool), 16, 16, 3,
                None) == K.KVQ_ERR_INVALID_ARG
    assert call("kv_quant_key_kitty_paged", ctypes.byref(cfg), ctypes.byref(paged), 0x1008, 8, 0, 0, 0, 0, None) == \
        K.KVQ_ERR_MISALIGNED                                           # 8 = ceil((1000 - 32) / 128) pages fit
    assert call("kv_quant_key_kitty_paged", ctypes.byref(cfg), ctypes.byref(paged), 16, 9, 0, 0, 0, 0, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert call("kv_quant_value_kitty_paged", ctypes.byref(cfg), ctypes.byref(paged), 16, 1, 0, 0, 2, None) == \
        K.KVQ_ERR_INVALID_ARG
    assert call("kv_release_kitty", ctypes.byref(cfg), ctypes.byref(dense), 0, ctypes.byref(pool), None) == \
        K.KVQ_ERR_INVALID_ARG


def test_decode_plan_and_workspace_checks(K):
    cfg = K.make_config()
    n, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, 32, 4096)
    assert n >= 1 and wsb >= 32 * 32 * n * 129 * 4
    n2, _ = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, 1, 131072)
    assert n2 <= 257
    cache = K.kvq_kivi_cache(32, 4096, 16, 16, 16, 16, 16, 16, 16)
    st = K.raw_call("kv_decode_attn", ctypes.byref(cfg), ctypes.byref(cache), 16, 16, 16, wsb - 1, None)
    assert st == K.KVQ_ERR_WORKSPACE
    st = K.raw_call("kv_decode_attn", ctypes.byref(cfg), ctypes.byref(cache), 16, 16, 0x1008, wsb, None)
    assert st == K.KVQ_ERR_MISALIGNED
    cache.k_sz = None
    st = K.raw_call("kv_decode_attn", ctypes.byref(cfg), ctypes.byref(cache), 16, 16, 16, wsb, None)
    assert st == K.KVQ_ERR_INVALID_ARG
    assert K.raw_call("kv_decode_attn_stage1", ctypes.byref(cfg), 7, ctypes.byref(cache), 16, 16, wsb,
                      None) == K.KVQ_ERR_INVALID_ARG


def test_segment_rules_agree_with_oracle(orc):
    from bit_kv_cache_keyquant_gb300 import cache as C
    for L in list(range(1, 700, 7)) + [4096, 32768, 131072]:
        assert C.kivi_segments(L, 128) == orc.kivi_segments(L, 128)
        assert C.kitty_segments(L, 128, 32, 128) == orc.kitty_segments(L, 128, 32, 128)
