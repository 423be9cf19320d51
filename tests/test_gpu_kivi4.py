"""GPU parity of the 4-bit KIVI widths (KIVI summary section 4: KIVI-4, and mixed K4V2 / K2V4) through
the C ABI: quantized bytes bit-exact against the oracle, attention within the oracle tolerance, and the
streaming append growing the same bytes as a bulk fill."""
import numpy as np
import pytest
import torch

from tests.gpu_util import assert_attn_close, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.fixture(scope="module")
def K():
    return lib()


def _data(rng, shape, kind):
    x = rng.standard_normal(shape)
    if kind == "outlier":
        x[..., 7] *= 40.0
    elif kind == "wide":
        x = x * 10.0 ** rng.uniform(-6, 4, shape[-1])
    return x.astype(np.float16)


@pytest.mark.parametrize("G", [32, 64, 128])
@pytest.mark.parametrize("kind", ["normal", "outlier", "wide"])
def test_quant_key_4bit_bitexact(K, orc, G, kind):
    rng = np.random.default_rng(400 + G)
    n = 29
    x = _data(rng, (n, G, D), kind)
    x[2, :, 5] = x[2, 0, 5]                          # a constant channel
    cfg = K.make_config(group_k=G, residual=128, bits_k=4)
    codes = torch.full((n, G * D // 2), 0xAB, dtype=torch.uint8, device=DEV)
    sz = torch.full((n, D), -1, dtype=torch.int32, device=DEV)
    K.kv_quant_key(cfg, torch.from_numpy(x).to(DEV), n, codes, sz)
    torch.cuda.synchronize()
    ref_codes, ref_sz = orc.kivi_quant_key(x, 4)
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    assert np.array_equal(sz.cpu().numpy().view(np.uint16).reshape(n, 2 * D), orc.kivi_key_sz_pack(ref_sz))


@pytest.mark.parametrize("Gv", [32, 64, 128])
@pytest.mark.parametrize("kind", ["normal", "outlier", "wide"])
def test_quant_value_4bit_bitexact(K, orc, Gv, kind):
    rng = np.random.default_rng(500 + Gv)
    n = 257
    x = _data(rng, (n, D), kind)
    # one query head per kv head: token-major; four (the grouped-query kernel, 4-bit values at Gv = 32):
    # 4-bit value tiles
    for Hq, Hkv in ((4, 4), (8, 2)):
        tiles = Hq // Hkv == 4 and Gv == 32
        cfg = K.make_config(group_v=Gv, bits_v=4, bits_k=4, n_q_heads=Hq, n_kv_heads=Hkv)
        rows = (n + 31) // 32 * 32 if tiles else n
        codes = torch.full((rows, D // 2), 0xAB, dtype=torch.uint8, device=DEV)
        sz = torch.full((n, D // Gv), -1, dtype=torch.int32, device=DEV)
        K.kv_quant_value(cfg, torch.from_numpy(x).to(DEV), n, codes, sz)
        torch.cuda.synchronize()
        ref_codes, ref_sz = orc.kivi_quant_value(x, Gv, 4, tiles=tiles)
        got = codes.cpu().numpy().reshape(-1)
        if tiles:
            written = np.zeros(got.size, bool)
            written[[orc.kivi_value_byte_offset4(t, c) for t in range(n) for c in range(64)]] = True
            assert np.array_equal(got[written], ref_codes.reshape(-1)[written])
            assert np.all(got[~written] == 0xAB)    # the last tile's bytes past token n are left unchanged
        else:
            assert np.array_equal(got, ref_codes.reshape(-1))
        assert np.array_equal(sz.cpu().numpy().view(np.uint16).reshape(n, D // Gv, 2), ref_sz)


def _fill(cfg, Ks, Vs, L_each, max_seq_len):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    c = C.KiviCache(cfg, B, max_seq_len, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            c.fill(b, h, torch.from_numpy(Ks[b][h][:L_each[b]]).to(DEV), torch.from_numpy(Vs[b][h][:L_each[b]]).to(DEV))
    return c


def _decode(K, cfg, c, q):
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, c.batch, c.max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((c.batch, cfg.n_q_heads, D), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn(cfg, c.desc(), torch.from_numpy(q).to(DEV), out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    return out.float().cpu().numpy()


def _oracle(orc, cfg, Ks, Vs, q, lens):
    g = cfg.n_q_heads // cfg.n_kv_heads
    out = np.zeros((len(lens), cfg.n_q_heads, D))
    for b, L in enumerate(lens):
        for h in range(cfg.n_kv_heads):
            parts = orc.kivi_build_one(Ks[b][h][:L], Vs[b][h][:L], cfg.group_k, cfg.group_v, cfg.residual,
                                       cfg.bits_k, cfg.bits_v)
            out[b, h * g:(h + 1) * g] = orc.kivi_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, G=cfg.group_k,
                                                            Gv=cfg.group_v, R=cfg.residual, bits_k=cfg.bits_k,
                                                            bits_v=cfg.bits_v)
    return out


@pytest.mark.parametrize("bk,bv", [(4, 4), (4, 2), (2, 4)])
@pytest.mark.parametrize("shape", [
    # (Hq, Hkv, lengths, G, Gv, R)
    (2, 2, [1, 33, 129, 700], 32, 32, 128),
    (4, 1, [1000, 1537], 64, 32, 128),        # grouped query heads, Gv = 32: tensor-core kernel at 4 bits
    (8, 2, [97, 2049], 32, 32, 128),
    (6, 2, [700, 1300], 128, 32, 256),        # 3 heads per kv head (one dead column pair)
    (4, 2, [800, 1100], 32, 64, 128),         # Gv = 64 at 4 bits: per-head kernel
    (2, 2, [640, 2000], 128, 128, 128),
    (3, 3, [900, 257], 32, 64, 64),
])
def test_decode_4bit_parity(K, orc, bk, bv, shape):
    Hq, Hkv, lens, G, Gv, R = shape
    rng = np.random.default_rng(sum(lens) + 10 * bk + bv + G)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=G, group_v=Gv, residual=R, bits_k=bk, bits_v=bv)
    gain = 1.0 + 19.0 * (rng.random(D) < 0.04)                 # a few x20 key channels
    Ks = [[(rng.standard_normal((L, D)) * gain).astype(np.float16) for _ in range(Hkv)] for L in lens]
    Vs = [[rng.standard_normal((L, D)).astype(np.float16) for _ in range(Hkv)] for L in lens]
    q = rng.standard_normal((len(lens), Hq, D)).astype(np.float16)
    c = _fill(cfg, Ks, Vs, lens, max(lens) + 5)
    assert_attn_close(_decode(K, cfg, c, q), _oracle(orc, cfg, Ks, Vs, q, lens))


@pytest.mark.parametrize("bk,bv", [(4, 4), (2, 4)])
def test_append_4bit_matches_fill(K, orc, bk, bv):
    rng = np.random.default_rng(90 + bk + bv)
    Hq, Hkv, G, Gv, R = 4, 2, 32, 32, 128
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=G, group_v=Gv, residual=R, bits_k=bk, bits_v=bv)
    L0, n = [120, 250], 150
    total = max(L0) + n
    Ks = [[rng.standard_normal((total, D)).astype(np.float16) for _ in range(Hkv)] for _ in range(2)]
    Vs = [[rng.standard_normal((total, D)).astype(np.float16) for _ in range(Hkv)] for _ in range(2)]
    grown = _fill(cfg, Ks, Vs, L0, total + 2)
    for step in range(n):
        kn = torch.from_numpy(np.stack([np.stack([Ks[b][h][L0[b] + step] for h in range(Hkv)]) for b in range(2)]))
        vn = torch.from_numpy(np.stack([np.stack([Vs[b][h][L0[b] + step] for h in range(Hkv)]) for b in range(2)]))
        K.kv_append_kivi(cfg, grown.desc(), kn.to(DEV), vn.to(DEV))
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    lens = [L + n for L in L0]
    full = _fill(cfg, Ks, Vs, lens, total + 2)
    from bit_kv_cache_keyquant_gb300.cache import kivi_segments
    for b, L in enumerate(lens):
        nkq, nvq = kivi_segments(L, R)
        assert torch.equal(grown.k_codes[b, :, :nkq // G], full.k_codes[b, :, :nkq // G])
        assert torch.equal(grown.k_sz[b, :, :nkq // G], full.k_sz[b, :, :nkq // G])
        assert torch.equal(grown.v_codes[b, :, :nvq], full.v_codes[b, :, :nvq])
        assert torch.equal(grown.v_sz[b, :, :nvq], full.v_sz[b, :, :nvq])
    q = rng.standard_normal((2, Hq, D)).astype(np.float16)
    a = _decode(K, cfg, grown, q)
    assert np.array_equal(a, _decode(K, cfg, full, q))
    assert_attn_close(a, _oracle(orc, cfg, Ks, Vs, q, lens))
