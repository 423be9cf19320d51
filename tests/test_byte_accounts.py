"""CPU checks of the algorithmic bytes that the bench divides by stage-1 time (the roofline numerator):
each cache's `nbytes_read` against the byte account of its stored format, written out here from the
formats themselves with the workloads' sizes (host tensors; no GPU, no kernel launch).

- KIVI (KIVI sections 3.1-3.3): b-bit codes, one fp16 (s, z) pair per channel per G-token key group and
  per Gv-channel value group of a token, fp16 residual of R tokens per side.
- Kitty ("Page-Centric Memory Layout"): a 128-token key page is 4096 B of low plane + 512 B of high plane
  (K = 16 boosted channels) + 128 B of boost index + 512 B of (s, z) = 5248 B; a value page is
  4096 B of codes + 512 B of (s, z) = 4608 B; sink, Q-buffers and local window stay fp16.
- WitCert INT8 (section 6.1 byte account): 129 B per token, head and side (128 code bytes + one fp16
  scale per channel per 256 tokens), the active block fp16.
"""
import pytest

D = 128


@pytest.fixture(scope="module")
def K():
    from bit_kv_cache_keyquant_gb300 import build
    build.build()
    from bit_kv_cache_keyquant_gb300 import kvq
    return kvq


def test_kivi_llama2_mha_layer(K):
    """B32, 32/32 heads, L4096, K2V2, G = Gv = 32, R = 128: 446,464 B per (row, head) of cache; with
    the fp16 query the stage-1 read is 457,441,280 B."""
    from bit_kv_cache_keyquant_gb300.cache import KiviCache
    cfg = K.make_config(n_q_heads=32, n_kv_heads=32)
    c = KiviCache(cfg, 1, 4096, device="cpu")
    quantized = 4096 - 128                      # both sides keep the last 128 tokens fp16 at L = 4096
    per_head = (2 * quantized * 128 // 4          # 2-bit codes, K and V: 126,976 B each
                + (quantized // 32) * 128 * 4     # key (s, z): 63,488 B
                + quantized * (128 // 32) * 4     # value (s, z): 63,488 B
                + 2 * 128 * 128 * 2)              # fp16 residual: 65,536 B
    assert per_head == 446464
    assert c.nbytes_read([4096]) == 32 * per_head
    assert 32 * c.nbytes_read([4096]) + 32 * 32 * 128 * 2 == 457441280


def test_kivi_tiny_and_4bit(K):
    from bit_kv_cache_keyquant_gb300.cache import KiviCache
    cfg = K.make_config(n_q_heads=4, n_kv_heads=4)
    c = KiviCache(cfg, 1, 512, device="cpu")
    # L512: 384 quantized tokens per side; plus q and o (512 B per head) the step moves 411,648 B
    assert c.nbytes_read([512]) == 4 * (2 * 384 * 32 + 12 * 512 + 384 * 16 + 65536)
    assert c.nbytes_read([512]) + 4 * 512 == 411648
    cfg4 = K.make_config(n_q_heads=32, n_kv_heads=32, bits_k=4, bits_v=4)
    c4 = KiviCache(cfg4, 1, 4096, device="cpu")
    assert c4.nbytes_read([4096]) == 32 * (2 * 3968 * 64 + 124 * 512 + 3968 * 16 + 65536)
    # residual boundary: at L = 513 the key residual holds 1 token, the value residual 128
    assert c.nbytes_read([513]) == 4 * ((512 * 32 + 16 * 512) + (385 * 32 + 385 * 16) + (1 + 128) * 256)


def test_kitty_mixed_key_layer(K):
    """L131072, S32 G128 R128, K = 16: 1023 key pages, 1022 value pages and 384 fp16 tokens per
    (row, kv head) (sink 2 x 32, key Q-buffer 96, value Q-buffer 96, local window 128)."""
    from bit_kv_cache_keyquant_gb300.cache import KittyCache
    cfg = K.make_config(n_q_heads=32, n_kv_heads=8, group_k=128, boost_k=16)
    assert K.kvq_kitty_key_page_bytes(cfg) == 4096 + 512 + 128 + 512 == 5248
    assert K.kvq_kitty_value_page_bytes(cfg) == 4096 + 512 == 4608
    c = KittyCache(cfg, 1, 131072, device="cpu")
    per_head = 1023 * 5248 + 1022 * 4608 + 384 * 128 * 2
    assert c.nbytes_read([131072]) == 8 * per_head
    # with q and o of the 16 x 32 query heads, the layer step of B16 moves 1302.8 MB
    total = 16 * c.nbytes_read([131072]) + 16 * 32 * 512
    assert round(total / 1e6, 1) == 1302.8
    cfg_pro = K.make_config(n_q_heads=32, n_kv_heads=8, group_k=128, boost_k=32)
    assert K.kvq_kitty_key_page_bytes(cfg_pro) == 4096 + 32 * 32 + 128 + 512
    # the high plane holds K rounded up to a multiple of 4 rows
    for Kb, rows in ((1, 4), (13, 16), (92, 92), (128, 128)):
        cfg_k = K.make_config(n_q_heads=32, n_kv_heads=8, group_k=128, boost_k=Kb)
        assert K.kvq_kitty_key_page_bytes(cfg_k) == 4096 + rows * 32 + 128 + 512


def test_int8_block_scale(K):
    from bit_kv_cache_keyquant_gb300.cache import Int8Cache
    cfg = K.make_config(n_q_heads=64, n_kv_heads=8)
    c = Int8Cache(cfg, 1, 16384 + 356, device="cpu")
    # 16384 + 356 tokens: 65 blocks of 256 quantized (129 B per token, head and side), 100 fp16
    assert c.nbytes_read([16384 + 356]) == 8 * 2 * (65 * 256 * 129 + 100 * 256)
    # an exact multiple of 256 keeps its last block fp16 (insert, attend, then quantize)
    assert c.nbytes_read([512]) == 8 * 2 * (256 * 129 + 256 * 256)
