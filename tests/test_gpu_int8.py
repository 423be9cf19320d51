"""GPU parity of the INT8 subtractive-dither decode path."""
import numpy as np
import pytest
import torch

from bit_kv_cache_keyquant_gb300 import inputs as I
from tests.gpu_util import assert_attn_close, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    return lib()


def _run(K, cfg, Ks, Vs, q, reqs, max_seq_len, layer, seed):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    cache = C.Int8Cache(cfg, B, max_seq_len, layer=layer, seed=seed, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            cache.fill(b, h, torch.from_numpy(Ks[b][h]).to(DEV), torch.from_numpy(Vs[b][h]).to(DEV), int(reqs[b]))
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8, B, max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((B, cfg.n_q_heads, 128), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_int8(cfg, cache.desc(), torch.from_numpy(q).to(DEV), out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    return out.float().cpu().numpy()


def _oracle(orc, cfg, Ks, Vs, q, reqs, layer, seed):
    g = cfg.n_q_heads // cfg.n_kv_heads
    B, Hkv = len(Ks), len(Ks[0])
    out = np.zeros((B, cfg.n_q_heads, 128))
    for b in range(B):
        for h in range(Hkv):
            L = Ks[b][h].shape[0]
            parts = orc.int8_build_one(Ks[b][h], Vs[b][h], seed, int(reqs[b]), layer, h)
            out[b, h * g:(h + 1) * g] = orc.int8_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, seed=seed,
                                                            request=int(reqs[b]), layer=layer, kv_head=h)
    return out


@pytest.mark.parametrize("Hq,Hkv,lens", [
    (8, 1, [1, 100, 256]),
    (8, 1, [257, 511, 700]),
    (6, 2, [1500, 300]),
    (2, 2, [1024, 999]),
])
def test_int8_decode_parity(K, orc, Hq, Hkv, lens):
    rng = np.random.default_rng(sum(lens) + Hq)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    Ks = [[(rng.standard_normal((L, 128)) * 10.0 ** rng.uniform(-1, 1, 128)).astype(np.float16) for _ in range(Hkv)]
          for L in lens]
    Vs = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(Hkv)] for L in lens]
    q = rng.standard_normal((len(lens), Hq, 128)).astype(np.float16)
    reqs = rng.integers(0, 2 ** 31 - 1, len(lens))
    layer, seed = 7, 0x0123456789ABCDEF
    got = _run(K, cfg, Ks, Vs, q, reqs, max(lens) + 3, layer, seed)
    assert_attn_close(got, _oracle(orc, cfg, Ks, Vs, q, reqs, layer, seed))


def test_int8_dither_dominated_parity(K, orc):
    """Cases whose outputs the dither moves far beyond the tolerance, so that a read side regenerating
    the wrong stream (K / V swapped, token index off by the block start, another head's tuple) fails by
    orders of magnitude: row 0 has K = 0 (uniform softmax: o = mean of the dequantized values over one
    quantized block and one fp16 token), row 1 large keys (a peaked softmax over two quantized blocks);
    values x100 make the dither part s * xi about 0.4 per element."""
    rng = np.random.default_rng(91)
    Hq, Hkv, lens = 8, 2, [257, 600]
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    Ks = [[np.zeros((257, 128), np.float16) for _ in range(Hkv)],
          [(rng.standard_normal((600, 128)) * 30).astype(np.float16) for _ in range(Hkv)]]
    Vs = [[(rng.standard_normal((L, 128)) * 100).astype(np.float16) for _ in range(Hkv)] for L in lens]
    q = rng.standard_normal((2, Hq, 128)).astype(np.float16)
    reqs = np.array([1234567, 89])
    layer, seed = 9, 0xFEDCBA9876543210
    want = _oracle(orc, cfg, Ks, Vs, q, reqs, layer, seed)
    got = _run(K, cfg, Ks, Vs, q, reqs, 600, layer, seed)
    assert_attn_close(got, want)
    # the same quantized cache read without its dither (x^ = s code) is far outside the tolerance
    g = Hq // Hkv
    parts = orc.int8_build_one(Ks[0][1], Vs[0][1], seed, int(reqs[0]), layer, 1)
    vs = np.array([[orc.half_to_double(int(x)) for x in parts[3][0]]])
    v_plain = np.concatenate([parts[1][:256].astype(np.float64) * vs, Vs[0][1][256:].astype(np.float64)])
    assert np.max(np.abs(v_plain.mean(axis=0) - want[0, g])) > 0.02


def test_int8_batch_order_invariance(K, orc):
    """Swapping batch rows together with their request ids swaps the outputs exactly."""
    rng = np.random.default_rng(77)
    cfg = K.make_config(n_q_heads=8, n_kv_heads=1)
    lens = [900, 600]
    Ks = [[rng.standard_normal((L, 128)).astype(np.float16)] for L in lens]
    Vs = [[rng.standard_normal((L, 128)).astype(np.float16)] for L in lens]
    q = rng.standard_normal((2, 8, 128)).astype(np.float16)
    reqs = np.array([11, 42])
    a = _run(K, cfg, Ks, Vs, q, reqs, 900, 3, 5)
    b = _run(K, cfg, Ks[::-1], Vs[::-1], q[::-1].copy(), reqs[::-1].copy(), 900, 3, 5)
    assert np.array_equal(a, b[::-1])


@pytest.mark.slow
def test_int8_workload_full_size_sampled(K, orc):
    """INT8 dither workload: B8, 64q/8kv, lengths U[16384, 65536]; sampled rows vs the oracle."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    w = I.WORKLOADS[5]
    cfg = K.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads)
    lens = I.seq_lens(w)
    reqs = I.request_ids(w)
    layer, seed = 5, w.seed
    Lmax = int(lens.max())
    cache = C.Int8Cache(cfg, w.batch, Lmax, layer=layer, seed=seed, device=DEV)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            L = int(lens[b])
            cache.fill(b, h, I.gen_kv_torch(w, I.T_K, b, h, L, DEV), I.gen_kv_torch(w, I.T_V, b, h, L, DEV),
                       int(reqs[b]))
    q = I.gen_q_torch(w, DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8, w.batch, Lmax)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty((w.batch, w.n_q_heads, 128), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_int8(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    qn = q.cpu().numpy()
    g = w.n_q_heads // w.n_kv_heads
    for b, h in ((0, 0), (w.batch - 1, w.n_kv_heads - 1), (3, 5)):
        L = int(lens[b])
        parts = orc.int8_build_one(I.gen_kv_np(w, I.T_K, b, h, L), I.gen_kv_np(w, I.T_V, b, h, L), seed,
                                   int(reqs[b]), layer, h)
        want = orc.int8_decode_one(qn[b, h * g:(h + 1) * g], *parts, L=L, seed=seed, request=int(reqs[b]),
                                   layer=layer, kv_head=h)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")
        # the int8 codes and scales written on the GPU are bit-exact
        assert np.array_equal(cache.k_codes[b, h, :256].cpu().numpy(), parts[0][:256])
        assert np.array_equal(cache.v_scale[b, h, 1].cpu().numpy().view(np.uint16), parts[3][1])


@pytest.mark.slow
def test_int8_offsets_beyond_2gib(K, orc):
    """Maximum-size addressing: int8 code arrays of 2.3 GB each (B16, 64 query / 16 kv heads, 69632 tokens).
    Random codes and scales fill every row; the first and the last (row, kv head) hold real data (the last
    at byte offsets beyond 2^31) and are checked against the oracle."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hq, Hkv, L = 16, 64, 16, 69632
    layer, seed = 2, 0x1234567890
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    cache = C.Int8Cache(cfg, B, L, layer=layer, seed=seed, device=DEV)
    assert (B * Hkv - 1) * L * 128 > 2 ** 31          # the last (row, kv head) starts past 2^31 bytes
    gen = torch.Generator(device=DEV).manual_seed(4)
    cache.k_codes.random_(-127, 128, generator=gen)
    cache.v_codes.random_(-127, 128, generator=gen)
    cache.k_scale.uniform_(0.0, 0.05, generator=gen)
    cache.v_scale.uniform_(0.0, 0.05, generator=gen)
    cache.k_tail.normal_(generator=gen)
    cache.v_tail.normal_(generator=gen)
    cache.seq_len.fill_(L)
    rng = np.random.default_rng(13)
    reqs = [11, 12]
    rows = {}
    for (b, h), rid in zip(((0, 0), (B - 1, Hkv - 1)), reqs):
        Kh = (rng.standard_normal((L, 128)) * 10.0 ** rng.uniform(-1, 1, 128)).astype(np.float16)
        Vh = rng.standard_normal((L, 128)).astype(np.float16)
        cache.fill(b, h, torch.from_numpy(Kh).to(DEV), torch.from_numpy(Vh).to(DEV), rid)
        rows[(b, h)] = (Kh, Vh, rid)
    q = torch.from_numpy(rng.standard_normal((B, Hq, 128)).astype(np.float16)).to(DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8, B, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_int8(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    assert np.isfinite(outn).all()
    g = Hq // Hkv
    for (b, h), (Kh, Vh, rid) in rows.items():
        parts = orc.int8_build_one(Kh, Vh, seed, rid, layer, h)
        want = orc.int8_decode_one(q[b, h * g:(h + 1) * g].cpu().numpy(), *parts, L=L, seed=seed, request=rid,
                                   layer=layer, kv_head=h)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")
