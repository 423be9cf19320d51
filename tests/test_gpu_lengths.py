"""Decode kernels against corrupt cached lengths (through the C ABI).

A seq_len outside [0, max_seq_len] is read clamped into that range, so that
no read leaves the caller's arrays, and KVQ_DEVICE_ERR_CAPACITY is recorded
in the device error flag.  A length above the capacity therefore decodes
exactly like a full row, a negative one like an empty row (zero output),
and the rows around them are untouched.
"""
import numpy as np
import pytest
import torch

from tests.gpu_util import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    return lib()


def _decode(K, fn, cfg, cache, variant, q):
    _, wsb = K.kv_decode_attn_plan(cfg, variant, cache.batch, cache.max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((cache.batch, cfg.n_q_heads, 128), float("nan"), dtype=torch.float16, device=DEV)
    fn(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    return out.cpu()


def _check(K, fn, cfg, cache, variant, q, Lmax):
    """Row 0 is full, row 1 holds Lmax // 3 tokens, row 2 is full: decode once as filled, then with row 0
    at Lmax + 1000 and row 2 at -5."""
    ref = _decode(K, fn, cfg, cache, variant, q)
    assert K.kvq_get_device_error() == 0
    good = cache.seq_len.clone()
    cache.seq_len[0] = Lmax + 1000
    cache.seq_len[2] = -5
    got = _decode(K, fn, cfg, cache, variant, q)
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_CAPACITY
    cache.seq_len.copy_(good)
    assert torch.equal(got[0], ref[0])                  # read as a full row
    assert torch.equal(got[1], ref[1])                  # untouched
    assert torch.count_nonzero(got[2]) == 0             # read as an empty row
    again = _decode(K, fn, cfg, cache, variant, q)      # the next call with sane lengths is clean
    assert K.kvq_get_device_error() == 0
    assert torch.equal(again, ref)


def _kv(rng, B, Hkv, lens, Lmax):
    return [[(torch.from_numpy(rng.standard_normal((lens[b], 128)).astype(np.float16)).to(DEV),
              torch.from_numpy(rng.standard_normal((lens[b], 128)).astype(np.float16)).to(DEV))
             for _ in range(Hkv)] for b in range(B)]


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2), (16, 2)])
def test_kivi_lengths_clamped(K, Hq, Hkv):
    from bit_kv_cache_keyquant_gb300 import cache as C
    rng = np.random.default_rng(3 + Hq)
    Lmax = 1100
    lens = [Lmax, Lmax // 3, Lmax]
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    cache = C.KiviCache(cfg, 3, Lmax, device=DEV)
    for b, row in enumerate(_kv(rng, 3, Hkv, lens, Lmax)):
        for h, (k, v) in enumerate(row):
            cache.fill(b, h, k, v)
    q = torch.from_numpy(rng.standard_normal((3, Hq, 128)).astype(np.float16)).to(DEV)
    _check(K, K.kv_decode_attn, cfg, cache, K.KVQ_VARIANT_KIVI, q, Lmax)


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2)])
def test_kitty_lengths_clamped(K, Hq, Hkv):
    from bit_kv_cache_keyquant_gb300 import cache as C
    rng = np.random.default_rng(13 + Hq)
    Lmax = 700
    lens = [Lmax, Lmax // 3, Lmax]
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, sink=32, residual=128, boost_k=16)
    cache = C.KittyCache(cfg, 3, Lmax, device=DEV)
    for b, row in enumerate(_kv(rng, 3, Hkv, lens, Lmax)):
        for h, (k, v) in enumerate(row):
            cache.fill(b, h, k, v)
    q = torch.from_numpy(rng.standard_normal((3, Hq, 128)).astype(np.float16)).to(DEV)
    _check(K, K.kv_decode_attn_kitty, cfg, cache, K.KVQ_VARIANT_KITTY, q, Lmax)


def test_int8_lengths_clamped(K):
    from bit_kv_cache_keyquant_gb300 import cache as C
    rng = np.random.default_rng(23)
    Lmax, Hq, Hkv = 900, 8, 2
    lens = [Lmax, Lmax // 3, Lmax]
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    cache = C.Int8Cache(cfg, 3, Lmax, layer=1, seed=7, device=DEV)
    for b, row in enumerate(_kv(rng, 3, Hkv, lens, Lmax)):
        for h, (k, v) in enumerate(row):
            cache.fill(b, h, k, v, 100 + b)
    q = torch.from_numpy(rng.standard_normal((3, Hq, 128)).astype(np.float16)).to(DEV)
    _check(K, K.kv_decode_attn_int8, cfg, cache, K.KVQ_VARIANT_INT8, q, Lmax)
