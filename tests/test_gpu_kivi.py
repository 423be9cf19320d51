"""GPU parity of the KIVI path and of Philox, through the C ABI.

Quantization (codes, (s, z)) must match the oracle bit for bit; attention
outputs within max-abs 2e-3 of the oracle's binary64 result (fp16 out,
fp32 accumulate).
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_keyquant_gb300 import inputs as I
from tests.gpu_util import assert_attn_close, curand_philox, lib, max_abs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    return lib()


def _rand_fp16(rng, shape, kind):
    if kind == "normal":
        x = rng.standard_normal(shape)
    elif kind == "outlier":
        x = rng.standard_normal(shape)
        x[..., 7] *= 40.0
    elif kind == "wide":
        x = rng.standard_normal(shape) * 10.0 ** rng.uniform(-6, 4, shape[-1])
    elif kind == "tiny":
        x = rng.standard_normal(shape) * 1e-6          # fp16 subnormals
    elif kind == "const":
        x = np.ones(shape) * 0.3
    else:
        raise ValueError(kind)
    return x.astype(np.float16)


@pytest.mark.parametrize("G", [32, 64, 128])
@pytest.mark.parametrize("kind", ["normal", "outlier", "wide", "tiny", "const"])
def test_quant_key_bitexact(K, orc, G, kind):
    rng = np.random.default_rng(100 + G)
    n = 37
    x = _rand_fp16(rng, (n, G, 128), kind)
    if kind == "normal":
        x[3, :, 11] = x[3, 0, 11]                    # a constant channel inside a group
        x[5, 2, 4] = np.float16(65504.0)
        x[5, 9, 4] = np.float16(-65504.0)            # widest fp16 range
    cfg = K.make_config(group_k=G, residual=128)
    xd = torch.from_numpy(x).to(DEV)
    codes = torch.full((n, G * 32), 0xAB, dtype=torch.uint8, device=DEV)
    sz = torch.full((n, 128), -1, dtype=torch.int32, device=DEV)
    K.kv_quant_key(cfg, xd, n, codes, sz)
    torch.cuda.synchronize()
    ref_codes, ref_sz = orc.kivi_quant_key(x)
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    assert np.array_equal(sz.cpu().numpy().view(np.uint16).reshape(n, 256), orc.kivi_key_sz_pack(ref_sz))


@pytest.mark.parametrize("Gv", [32, 64, 128])
@pytest.mark.parametrize("kind", ["normal", "outlier", "wide", "tiny", "const"])
def test_quant_value_bitexact(K, orc, Gv, kind):
    rng = np.random.default_rng(200 + Gv)
    n = 333
    x = _rand_fp16(rng, (n, 128), kind)
    for Hq, Hkv in ((4, 4), (8, 2)):                # one query head per kv head: token-major; four: value tiles
        tiles = Hq // Hkv == 4
        cfg = K.make_config(group_v=Gv, n_q_heads=Hq, n_kv_heads=Hkv)
        xd = torch.from_numpy(x).to(DEV)
        rows = (n + 31) // 32 * 32 if tiles else n  # whole 32-token value tiles
        codes = torch.full((rows, 32), 0xAB, dtype=torch.uint8, device=DEV)
        sz = torch.full((n, 128 // Gv), -1, dtype=torch.int32, device=DEV)
        K.kv_quant_value(cfg, xd, n, codes, sz)
        torch.cuda.synchronize()
        ref_codes, ref_sz = orc.kivi_quant_value(x, Gv, tiles=tiles)
        got = codes.cpu().numpy().reshape(-1)
        if tiles:
            written = np.zeros(got.size, bool)
            written[[orc.kivi_value_byte_offset(t, c) for t in range(n) for c in range(0, 128, 4)]] = True
            assert np.array_equal(got[written], ref_codes.reshape(-1)[written])
            assert np.all(got[~written] == 0xAB)    # the last tile's bytes past token n are left unchanged
        else:
            assert np.array_equal(got, ref_codes.reshape(-1))
        assert np.array_equal(sz.cpu().numpy().view(np.uint16).reshape(n, 128 // Gv, 2), ref_sz)


def _run_decode(K, cfg, Ks, Vs, q, max_seq_len):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    cache = C.KiviCache(cfg, B, max_seq_len, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            cache.fill(b, h, torch.from_numpy(Ks[b][h]).to(DEV), torch.from_numpy(Vs[b][h]).to(DEV))
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)            # poisoned workspace
    out = torch.full((B, cfg.n_q_heads, 128), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn(cfg, cache.desc(), torch.from_numpy(q).to(DEV), out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    return out.float().cpu().numpy()


def _oracle_decode(orc, cfg, Ks, Vs, q):
    g = cfg.n_q_heads // cfg.n_kv_heads
    B, Hkv = len(Ks), len(Ks[0])
    out = np.zeros((B, cfg.n_q_heads, 128))
    for b in range(B):
        for h in range(Hkv):
            L = Ks[b][h].shape[0]
            parts = orc.kivi_build_one(Ks[b][h], Vs[b][h], cfg.group_k, cfg.group_v, cfg.residual)
            out[b, h * g:(h + 1) * g] = orc.kivi_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, G=cfg.group_k,
                                                            Gv=cfg.group_v, R=cfg.residual)
    return out


@pytest.mark.parametrize("shape", [
    # (B, Hq, Hkv, lengths, G, Gv, R)
    (3, 2, 2, [1, 33, 129], 32, 32, 128),
    (2, 4, 1, [300, 1000], 32, 32, 128),
    (2, 8, 2, [511, 512], 32, 32, 128),
    (2, 2, 2, [640, 1537], 64, 32, 128),
    (1, 2, 1, [2000], 128, 128, 128),
    (2, 2, 2, [700, 900], 32, 64, 64),
    (1, 1, 1, [128], 32, 32, 128),
    (1, 1, 1, [4095], 32, 32, 256),
    # grouped-query tensor-core kernel: 3 heads (one dead B column pair), Gv = 64 and 128
    (3, 6, 2, [97, 1024, 1333], 32, 32, 128),
    (2, 4, 2, [700, 1900], 32, 64, 64),
    (1, 8, 4, [1025], 64, 128, 128),
    # 8 and 6 query heads per kv head: two grouped-query units per kv head (64q/8kv: Llama-3-70B-shaped)
    (1, 8, 1, [1200], 32, 32, 128),
    (2, 12, 2, [700, 1900], 32, 32, 128),
    (1, 64, 8, [1100], 32, 32, 128),
])
def test_decode_parity_small(K, orc, shape):
    B, Hq, Hkv, lens, G, Gv, R = shape
    rng = np.random.default_rng(sum(lens) + Hq)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=G, group_v=Gv, residual=R)
    Ks = [[(rng.standard_normal((lens[b], 128)) * (1 + 9 * (rng.random(128) < 0.03))).astype(np.float16)
           for _ in range(Hkv)] for b in range(B)]
    Vs = [[rng.standard_normal((lens[b], 128)).astype(np.float16) for _ in range(Hkv)] for b in range(B)]
    q = rng.standard_normal((B, Hq, 128)).astype(np.float16)
    got = _run_decode(K, cfg, Ks, Vs, q, max(lens) + 5)
    want = _oracle_decode(orc, cfg, Ks, Vs, q)
    assert_attn_close(got, want)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_decode_wide_outlier_channels(K, orc, Hq, Hkv):
    """Key channels x20 and a large query (the logit scale of the tiny workload): the fp16 hi / lo
    key weights of the tensor-core path and the fixed-point dp4a key products of the per-head path both hold."""
    rng = np.random.default_rng(Hq * 31 + Hkv)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    lens = [777, 2048]
    gain = np.ones(128)
    gain[[3, 40, 77, 120]] = 20.0
    Ks = [[(rng.standard_normal((L, 128)) * gain).astype(np.float16) for _ in range(Hkv)] for L in lens]
    Vs = [[(rng.standard_normal((L, 128)) * 3.0).astype(np.float16) for _ in range(Hkv)] for L in lens]
    q = (rng.standard_normal((2, Hq, 128)) * 2.0).astype(np.float16)
    got = _run_decode(K, cfg, Ks, Vs, q, 2048)
    assert_attn_close(got, _oracle_decode(orc, cfg, Ks, Vs, q))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
@pytest.mark.parametrize("case", ["zero_query", "wide_channels", "const_groups", "huge_query", "big_query"])
def test_decode_key_weight_extremes(K, orc, Hq, Hkv, case):
    """Key weights alpha q s at the edges of the per-head kernel's fixed-point form (one power-of-two
    scale per 32-token group, set by the group's largest |weight|) and of the tensor-core hi / lo
    split: an all-zero query (every weight 0), channel ranges from 1e-4 to 3e4 in one group, groups
    whose channels are constant (s = 0), and a query of +-300 in one channel over channels of about
    0.02, a range of 2^14 (the grouped-query path keeps every channel's weight a normal fp16 number
    up to that range; beyond it the smallest channels fall to fp16 subnormals and lose their key
    contributions, and the logits' ties on the large channel are then broken without them), and a query of
    +-3000 in one channel over channels of about 1e-3 (logits of about 800: the 2-bit codes tie many tokens on
    the large channel and the small channels break the ties; beyond about 1e4 over 1e-3 even an fp32
    accumulation of exact products misses 2e-3, see test_oracle_pins.py)."""
    rng = np.random.default_rng({"zero_query": 11, "wide_channels": 12, "const_groups": 13, "huge_query": 14,
                                 "big_query": 15}[case] + Hq)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    lens = [700, 1300]
    Ks, Vs = [], []
    for L in lens:
        kr, vr = [], []
        for _ in range(Hkv):
            k = rng.standard_normal((L, 128))
            if case == "wide_channels":
                k = np.clip(k * 10.0 ** rng.uniform(-4, 4.4, 128), -6.0e4, 6.0e4)
            if case == "const_groups":
                for g0 in range(0, L - 31, 64):                    # every other 32-token group constant
                    k[g0:g0 + 32] = k[g0]
            kr.append(k.astype(np.float16))
            vr.append(rng.standard_normal((L, 128)).astype(np.float16))
        Ks.append(kr)
        Vs.append(vr)
    q = rng.standard_normal((2, Hq, 128))
    if case == "zero_query":
        q[0, 0] = 0.0
        q[1, :] = 0.0
    if case == "wide_channels":
        q *= 10.0 ** rng.uniform(-3, 2, 128)
    if case == "huge_query":
        q *= 0.02
        q[:, :, 5] = 300.0
        q[1, 0, 5] = -300.0
    if case == "big_query":
        q *= 1e-3
        q[:, :, 5] = 3000.0
        q[1, 0, 5] = -3000.0
    q = q.astype(np.float16)
    got = _run_decode(K, cfg, Ks, Vs, q, 1300)
    assert np.isfinite(got).all()
    assert_attn_close(got, _oracle_decode(orc, cfg, Ks, Vs, q))


def test_decode_capacity_and_split_invariance(K, orc):
    """The same cache content under a larger capacity (more splits) gives the same result."""
    rng = np.random.default_rng(7)
    cfg = K.make_config(n_q_heads=4, n_kv_heads=2)
    lens = [1500, 700]
    Ks = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(2)] for L in lens]
    Vs = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(2)] for L in lens]
    q = rng.standard_normal((2, 4, 128)).astype(np.float16)
    a = _run_decode(K, cfg, Ks, Vs, q, 1500)
    b = _run_decode(K, cfg, Ks, Vs, q, 9000)
    assert max_abs(a, b) <= 1e-3
    assert_attn_close(a, _oracle_decode(orc, cfg, Ks, Vs, q))


def test_decode_residual_only_matches_sdpa(K):
    """L <= R: nothing is quantized, the kernel is plain attention (torch SDPA, fp32)."""
    rng = np.random.default_rng(8)
    cfg = K.make_config(n_q_heads=8, n_kv_heads=2)
    L = 100
    Ks = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(2)]]
    Vs = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(2)]]
    q = rng.standard_normal((1, 8, 128)).astype(np.float16)
    got = _run_decode(K, cfg, Ks, Vs, q, 256)
    kt = torch.from_numpy(np.stack(Ks[0])).float().repeat_interleave(4, 0)[None]
    vt = torch.from_numpy(np.stack(Vs[0])).float().repeat_interleave(4, 0)[None]
    qt = torch.from_numpy(q).float()[:, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, :, 0].numpy()
    assert_attn_close(got, ref)


def test_workload1_tiny_full(K, orc):
    """Tiny K2V2 workload: B=1, 4 MHA heads, 512 tokens, 4 key channels x20; every output."""
    w = I.WORKLOADS[1]
    cfg = K.make_config(n_q_heads=4, n_kv_heads=4)
    Ks = [[I.gen_kv_np(w, I.T_K, 0, h, w.seq_len) for h in range(4)]]
    Vs = [[I.gen_kv_np(w, I.T_V, 0, h, w.seq_len) for h in range(4)]]
    q = I.gen_q_np(w)
    got = _run_decode(K, cfg, Ks, Vs, q, w.seq_len)
    assert_attn_close(got, _oracle_decode(orc, cfg, Ks, Vs, q))


@pytest.mark.slow
@pytest.mark.parametrize("widx", [2, 3])
def test_workload_full_size_sampled(K, orc, widx):
    """Full Llama-2-7B / Llama-3-8B shapes, the launch bench.py times; sampled (b, h) rows vs the oracle."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    w = I.WORKLOADS[widx]
    cfg = K.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads)
    L = w.seq_len
    cache = C.KiviCache(cfg, w.batch, L, device=DEV)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            cache.fill(b, h, I.gen_kv_torch(w, I.T_K, b, h, L, DEV), I.gen_kv_torch(w, I.T_V, b, h, L, DEV))
    q = I.gen_q_torch(w, DEV)
    n, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, w.batch, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty((w.batch, w.n_q_heads, 128), dtype=torch.float16, device=DEV)
    K.kv_decode_attn(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    assert np.isfinite(outn).all()
    qn = q.cpu().numpy()
    g = w.n_q_heads // w.n_kv_heads
    rng = np.random.default_rng(widx)
    for b, h in {(0, 0), (w.batch - 1, w.n_kv_heads - 1), *[(int(rng.integers(w.batch)), int(rng.integers(w.n_kv_heads))) for _ in range(3)]}:
        parts = orc.kivi_build_one(I.gen_kv_np(w, I.T_K, b, h, L), I.gen_kv_np(w, I.T_V, b, h, L))
        want = orc.kivi_decode_one(qn[b, h * g:(h + 1) * g], *parts, L=L)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")
    # quantized codes of a sampled group are bit-exact at full size too
    kc, ksz = orc.kivi_quant_key(I.gen_kv_np(w, I.T_K, 1, 0, 64)[None, :32])
    assert np.array_equal(cache.k_codes[1, 0, 0].cpu().numpy(), kc[0])
    assert np.array_equal(cache.k_sz[1, 0, 0].cpu().numpy().view(np.uint16), orc.kivi_key_sz_pack(ksz)[0])


@pytest.mark.slow
@pytest.mark.parametrize("widx", [2, 3, 9, 10])
def test_workload_shapes_gaussian_sampled(K, orc, widx):
    """The workloads' head counts, code widths and full lengths with Gaussian activations (N(0, 1)
    rounded to fp16, one key channel per kv head scaled by 15): the tails and off-grid values that the
    workload generator's bounded grid never produces.  Two batch rows; sampled (row, kv head) pairs
    against the oracle, in the launch shape of the full workload's kernel."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    w = I.WORKLOADS[widx]
    B, L, Hkv = 2, w.seq_len, w.n_kv_heads
    cfg = K.make_config(n_q_heads=w.n_q_heads, n_kv_heads=Hkv, bits_k=w.bits_k, bits_v=w.bits_v)
    rng = np.random.default_rng(1000 + widx)
    pairs = {(0, 0), (1, Hkv - 1), (0, Hkv // 2)}
    cache = C.KiviCache(cfg, B, L, device=DEV)
    kept = {}
    for b in range(B):
        for h in range(Hkv):
            k = rng.standard_normal((L, 128), dtype=np.float32)
            k[:, (7 * h + 3) % 128] *= 15.0
            Kh = k.astype(np.float16)
            Vh = rng.standard_normal((L, 128), dtype=np.float32).astype(np.float16)
            cache.fill(b, h, torch.from_numpy(Kh).to(DEV), torch.from_numpy(Vh).to(DEV))
            if (b, h) in pairs:
                kept[(b, h)] = (Kh, Vh)
    q = torch.from_numpy(rng.standard_normal((B, w.n_q_heads, 128), dtype=np.float32).astype(np.float16)).to(DEV)
    n, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty((B, w.n_q_heads, 128), dtype=torch.float16, device=DEV)
    K.kv_decode_attn(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    assert np.isfinite(outn).all()
    qn = q.cpu().numpy()
    g = w.n_q_heads // Hkv
    for (b, h), (Kh, Vh) in kept.items():
        parts = orc.kivi_build_one(Kh, Vh, bits_k=w.bits_k, bits_v=w.bits_v)
        want = orc.kivi_decode_one(qn[b, h * g:(h + 1) * g], *parts, L=L, bits_k=w.bits_k, bits_v=w.bits_v)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")


@pytest.mark.slow
def test_decode_offsets_beyond_2gib(K, orc):
    """Maximum-size addressing: a cache whose code and parameter arrays span 4.3 GB (B32, 64 query / 16 kv
    heads, 262144 tokens).  Random bytes fill every row; the first and the last (row, kv head) hold real
    data (the last at byte offsets far beyond 2^31) and are checked against the oracle."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hq, Hkv, L = 32, 64, 16, 262144
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    cache = C.KiviCache(cfg, B, L, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(5)
    cache.k_codes.random_(0, 256, generator=gen)
    cache.v_codes.random_(0, 256, generator=gen)
    cache.k_sz.view(torch.float16).uniform_(0.0, 0.25, generator=gen)
    cache.v_sz.view(torch.float16).uniform_(0.0, 0.25, generator=gen)
    cache.k_res.normal_(generator=gen)
    cache.v_res.normal_(generator=gen)
    cache.seq_len.fill_(L)
    assert (B * Hkv - 1) * L * 32 > 2 ** 31          # the last (row, kv head) starts past 2^31 bytes
    rng = np.random.default_rng(9)
    rows = {}
    for b, h in ((0, 0), (B - 1, Hkv - 1)):
        Kh = (rng.standard_normal((L, 128)) * (1 + 9 * (rng.random(128) < 0.02))).astype(np.float16)
        Vh = rng.standard_normal((L, 128)).astype(np.float16)
        cache.fill(b, h, torch.from_numpy(Kh).to(DEV), torch.from_numpy(Vh).to(DEV))
        rows[(b, h)] = (Kh, Vh)
    q = torch.from_numpy(rng.standard_normal((B, Hq, 128)).astype(np.float16)).to(DEV)
    n, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    assert np.isfinite(outn).all()
    g = Hq // Hkv
    for (b, h), (Kh, Vh) in rows.items():
        want = orc.kivi_decode_one(q[b, h * g:(h + 1) * g].cpu().numpy(), *orc.kivi_build_one(Kh, Vh), L=L)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")


# ---------------------------------------------------------------------------
# Philox
# ---------------------------------------------------------------------------
def _philox_cases():
    rng = np.random.default_rng(5)
    ctr = [[0, 0, 0, 0], [0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF], [0x80000000, 0, 0xFFFFFFFF, 1],
           [12345, 3, 0x00020007, 99]]
    key = [[0, 0], [0xFFFFFFFF, 0xFFFFFFFF], [0xDEADBEEF, 0x80000000], [1, 2]]
    ctr += rng.integers(0, 2 ** 32, (60, 4), dtype=np.uint64).tolist()
    key += rng.integers(0, 2 ** 32, (60, 2), dtype=np.uint64).tolist()
    return np.array(ctr, np.uint32), np.array(key, np.uint32)


def test_philox_matches_oracle(K, orc):
    ctr, key = _philox_cases()
    n = len(ctr)
    out = torch.zeros((n, 4), dtype=torch.int32, device=DEV)
    K.kvq_philox4x32_10(torch.from_numpy(ctr.view(np.int32)).to(DEV), torch.from_numpy(key.view(np.int32)).to(DEV), n,
                        out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    for i in range(n):
        assert np.array_equal(got[i], orc.philox(ctr[i], key[i])), i


def test_philox_oracle_matches_curand(orc):
    """Independent known answers: cuRAND's Philox4x32-10 at the same raw counter and key."""
    ctr, key = _philox_cases()
    ctr[:, 1] &= 0x3FFFFFFF                # curand_init's offset = 4 * (ctr0 | ctr1 << 32) must fit 64 bits
    n = len(ctr)
    c = torch.from_numpy(ctr.view(np.int32)).to(DEV)
    k = torch.from_numpy(key.view(np.int32)).to(DEV)
    out = torch.zeros((n, 4), dtype=torch.int32, device=DEV)
    assert curand_philox().curand_philox_ref(c.data_ptr(), k.data_ptr(), n, out.data_ptr()) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    for i in range(n):
        assert np.array_equal(got[i], orc.philox(ctr[i], key[i])), i
