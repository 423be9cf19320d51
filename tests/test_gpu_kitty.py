"""GPU parity of the Kitty decode path (pages quantized on the GPU, attention
vs the oracle's binary64 result, max-abs 2e-3)."""
import numpy as np
import pytest
import torch

from bit_kv_cache_keyquant_gb300 import inputs as I
from tests.gpu_util import assert_attn_close, lib, max_abs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    return lib()


def _run(K, cfg, Ks, Vs, q, max_seq_len, score_mode=0):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    cache = C.KittyCache(cfg, B, max_seq_len, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            cache.fill(b, h, torch.from_numpy(Ks[b][h]).to(DEV), torch.from_numpy(Vs[b][h]).to(DEV), score_mode)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KITTY, B, max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((B, cfg.n_q_heads, 128), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_kitty(cfg, cache.desc(), torch.from_numpy(q).to(DEV), out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    return out.float().cpu().numpy()


def _oracle(orc, cfg, Ks, Vs, q, score_mode=0):
    g = cfg.n_q_heads // cfg.n_kv_heads
    B, Hkv = len(Ks), len(Ks[0])
    out = np.zeros((B, cfg.n_q_heads, 128))
    for b in range(B):
        for h in range(Hkv):
            L = Ks[b][h].shape[0]
            parts = orc.kitty_build_one(Ks[b][h], Vs[b][h], 128, cfg.boost_k, cfg.sink, cfg.residual, score_mode)
            out[b, h * g:(h + 1) * g] = orc.kitty_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, K=cfg.boost_k,
                                                             S=cfg.sink, R=cfg.residual)
    return out


@pytest.mark.parametrize("lens,Kb,mode,Hq,Hkv", [
    ([1, 20, 33], 16, 0, 8, 2),
    ([161, 288, 416], 16, 0, 8, 2),
    ([417, 700, 2000], 16, 0, 8, 2),
    ([1500, 3000], 32, 0, 8, 2),
    ([1500, 2222], 16, 1, 8, 2),
    ([900, 1300], 0, 0, 8, 2),
    ([1700], 48, 0, 8, 2),          # three boosted k-steps
    ([1300], 92, 0, 4, 2),          # the largest supported boost
    ([1300], 13, 0, 8, 2),          # K not a multiple of 4: a padded row group, a partial k-step
    ([1100], 21, 1, 2, 2),          # the same on the per-head kernel (two high k-steps)
    ([1250], 90, 0, 8, 2),          # six high k-steps, two padded rows
    ([800, 1900], 16, 0, 6, 2),     # three heads per kv head (one dead tensor-core column pair)
    ([600, 1400], 16, 0, 2, 2),     # one head per kv head: per-head kernel
    ([1234], 16, 0, 8, 1),          # eight heads per kv head: two grouped-query units per kv head
    ([1500], 16, 0, 12, 2),         # six heads per kv head
    ([900], 16, 0, 64, 8),          # 64q/8kv
])
def test_kitty_decode_parity(K, orc, lens, Kb, mode, Hq, Hkv):
    rng = np.random.default_rng(sum(lens) + Kb + mode + Hq)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, sink=32, residual=128, boost_k=Kb)
    sig = 10.0 ** rng.uniform(-0.3, 0.9, (Hkv, 128))
    Ks = [[(rng.standard_normal((L, 128)) * sig[h]).astype(np.float16) for h in range(Hkv)] for L in lens]
    Vs = [[rng.standard_normal((L, 128)).astype(np.float16) for h in range(Hkv)] for L in lens]
    q = rng.standard_normal((len(lens), Hq, 128)).astype(np.float16)
    got = _run(K, cfg, Ks, Vs, q, max(lens) + 7, mode)
    want = _oracle(orc, cfg, Ks, Vs, q, mode)
    assert_attn_close(got, want)


@pytest.mark.slow
def test_kitty_workload_full_size_sampled(K, orc):
    """Qwen3-8B-shaped mixed key workload (B16, 32q/8kv, L=131072); sampled rows vs the oracle."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    w = I.WORKLOADS[4]
    cfg = K.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, group_k=128, sink=32, residual=128,
                        boost_k=16)
    L = w.seq_len
    cache = C.KittyCache(cfg, w.batch, L, device=DEV)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            cache.fill(b, h, I.gen_kv_torch(w, I.T_K, b, h, L, DEV), I.gen_kv_torch(w, I.T_V, b, h, L, DEV))
    q = I.gen_q_torch(w, DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KITTY, w.batch, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty((w.batch, w.n_q_heads, 128), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_kitty(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    assert np.isfinite(outn).all()
    qn = q.cpu().numpy()
    g = w.n_q_heads // w.n_kv_heads
    for b, h in ((0, 0), (w.batch - 1, w.n_kv_heads - 1), (7, 3)):
        Kn = I.gen_kv_np(w, I.T_K, b, h, L)
        Vn = I.gen_kv_np(w, I.T_V, b, h, L)
        parts = orc.kitty_build_one(Kn, Vn)
        want = orc.kitty_decode_one(qn[b, h * g:(h + 1) * g], *parts, L=L)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")
        # the key pages written on the GPU are bit-exact too
        assert np.array_equal(cache.k_pages[b, h, 5].cpu().numpy(), parts[0][5])


@pytest.mark.slow
@pytest.mark.parametrize("mode", [0, 1])
def test_kitty_workload_shape_gaussian_sampled(K, orc, mode):
    """The mixed-key workload's heads and full length with Gaussian activations (per-channel sigma
    log-uniform over [0.5, 8], as the workload states its key channels): two batch rows, both boost
    selections, sampled (row, kv head) pairs against the oracle."""
    w = I.WORKLOADS[4]
    B, L, Hkv = 2, w.seq_len, w.n_kv_heads
    cfg = K.make_config(n_q_heads=w.n_q_heads, n_kv_heads=Hkv, group_k=128, sink=32, residual=128, boost_k=16)
    rng = np.random.default_rng(4000 + mode)
    sig = 2.0 ** rng.uniform(-1.0, 3.0, (Hkv, 128))
    Ks = [[(rng.standard_normal((L, 128), dtype=np.float32) * sig[h]).astype(np.float16) for h in range(Hkv)]
          for _ in range(B)]
    Vs = [[rng.standard_normal((L, 128), dtype=np.float32).astype(np.float16) for h in range(Hkv)] for _ in range(B)]
    q = rng.standard_normal((B, w.n_q_heads, 128), dtype=np.float32).astype(np.float16)
    got = _run(K, cfg, Ks, Vs, q, L, mode)
    g = w.n_q_heads // Hkv
    for b, h in ((0, 0), (1, Hkv - 1), (0, Hkv // 2)):
        parts = orc.kitty_build_one(Ks[b][h], Vs[b][h], 128, 16, 32, 128, mode)
        want = orc.kitty_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, K=16, S=32, R=128)
        assert_attn_close(got[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")


@pytest.mark.slow
def test_kitty_offsets_beyond_2gib(K, orc):
    """Maximum-size addressing: key page records spanning 2.2 GB (B32, 64 query / 16 kv heads, 104992 tokens).
    Random bytes fill every page; the first and the last (row, kv head) hold real data (the last at byte
    offsets beyond 2^31) and are checked against the oracle."""
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hq, Hkv, L = 32, 64, 16, 32 + 820 * 128
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, sink=32, residual=128, boost_k=16)
    cache = C.KittyCache(cfg, B, L, device=DEV)
    assert (B * Hkv - 1) * 820 * cache.kpb > 2 ** 31   # the last (row, kv head) starts past 2^31 bytes
    gen = torch.Generator(device=DEV).manual_seed(3)
    # random codes; s, z of every page set to small fp16 values; idx left 0 (boost rank 0)
    cache.k_pages.random_(0, 256, generator=gen)
    cache.v_pages.random_(0, 256, generator=gen)
    kpb, vpb = cache.kpb, cache.vpb
    cache.k_pages[..., kpb - 512:].view(torch.float16).uniform_(0.0, 0.2, generator=gen)
    cache.k_pages[..., kpb - 512 - 128:kpb - 512].fill_(17)            # idx: no channel boosted
    cache.v_pages[..., vpb - 512:].view(torch.float16).uniform_(0.0, 0.2, generator=gen)
    for t in (cache.k_sink, cache.v_sink, cache.k_qbuf, cache.v_qbuf, cache.v_local):
        t.normal_(generator=gen)
    cache.seq_len.fill_(L)
    rng = np.random.default_rng(12)
    rows = {}
    for b, h in ((0, 0), (B - 1, Hkv - 1)):
        sig = 0.5 * 16.0 ** rng.random(128)
        Kh = (rng.standard_normal((L, 128)) * sig).astype(np.float16)
        Vh = rng.standard_normal((L, 128)).astype(np.float16)
        cache.fill(b, h, torch.from_numpy(Kh).to(DEV), torch.from_numpy(Vh).to(DEV))
        rows[(b, h)] = (Kh, Vh)
    q = torch.from_numpy(rng.standard_normal((B, Hq, 128)).astype(np.float16)).to(DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KITTY, B, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_kitty(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    outn = out.float().cpu().numpy()
    assert np.isfinite(outn).all()
    g = Hq // Hkv
    for (b, h), (Kh, Vh) in rows.items():
        parts = orc.kitty_build_one(Kh, Vh)
        want = orc.kitty_decode_one(q[b, h * g:(h + 1) * g].cpu().numpy(), *parts, L=L)
        assert_attn_close(outn[b, h * g:(h + 1) * g], want, f"row {b}, kv head {h}")


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2)])
def test_kitty_decode_big_query(K, orc, Hq, Hkv):
    """A query of +-3000 in one channel over channels of about 1e-3 (logits of about 800; ties on the large
    channel broken by the small ones) on the per-head and the grouped-query Kitty kernels."""
    rng = np.random.default_rng(70 + Hq)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, sink=32, residual=128, boost_k=16)
    lens = [700, 1300]
    Ks = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(Hkv)] for L in lens]
    Vs = [[rng.standard_normal((L, 128)).astype(np.float16) for _ in range(Hkv)] for L in lens]
    q = rng.standard_normal((2, Hq, 128)) * 1e-3
    q[:, :, 5] = 3000.0
    q[1, 0, 5] = -3000.0
    q = q.astype(np.float16)
    got = _run(K, cfg, Ks, Vs, q, 1300)
    assert_attn_close(got, _oracle(orc, cfg, Ks, Vs, q))
