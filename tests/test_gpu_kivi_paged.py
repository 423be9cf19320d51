"""GPU parity of the paged KIVI cache: pages of 128 tokens from a shared pool through a per-request page
table.  The same tokens decode bit-identically from the dense and the paged cache (the same kernels and
arithmetic, only the addressing differs), match the oracle, and grow by streaming append into pages
taken from the free stack."""
import numpy as np
import pytest
import torch

from bit_kv_cache_keyquant_gb300.cache import kivi_segments
from tests.gpu_util import assert_attn_close, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.fixture(scope="module")
def K():
    return lib()


def _paged(cfg, Ks, Vs, lens, max_seq_len, n_pages, seed=None):
    from bit_kv_cache_keyquant_gb300 import cache as C
    c = C.KiviPagedCache(cfg, len(lens), max_seq_len, n_pages, device=DEV)
    if seed is not None:
        c.shuffle_free(np.random.default_rng(seed).permutation(n_pages))
    for b, L in enumerate(lens):
        if L:
            c.fill(b, torch.from_numpy(np.stack([k[:L] for k in Ks[b]])).to(DEV),
                   torch.from_numpy(np.stack([v[:L] for v in Vs[b]])).to(DEV))
    return c


def _dense(cfg, Ks, Vs, lens, max_seq_len):
    from bit_kv_cache_keyquant_gb300 import cache as C
    c = C.KiviCache(cfg, len(lens), max_seq_len, device=DEV)
    for b, L in enumerate(lens):
        for h in range(cfg.n_kv_heads):
            c.fill(b, h, torch.from_numpy(Ks[b][h][:L]).to(DEV), torch.from_numpy(Vs[b][h][:L]).to(DEV))
    return c


def _decode(K, cfg, c, q, paged):
    variant = K.KVQ_VARIANT_KIVI_PAGED if paged else K.KVQ_VARIANT_KIVI
    _, wsb = K.kv_decode_attn_plan(cfg, variant, c.batch, c.max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((c.batch, cfg.n_q_heads, D), float("nan"), dtype=torch.float16, device=DEV)
    qd = torch.from_numpy(q).to(DEV) if isinstance(q, np.ndarray) else q
    if paged:
        K.kv_decode_attn_kivi_paged(cfg, c.desc(), qd, out, ws, wsb)
    else:
        K.kv_decode_attn(cfg, c.desc(), qd, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    return out


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


def _data(rng, lens, Hkv, total=None):
    total = total or max(lens)
    gain = 1.0 + 9.0 * (rng.random(D) < 0.05)
    Ks = [[(rng.standard_normal((total, D)) * gain).astype(np.float16) for _ in range(Hkv)] for _ in lens]
    Vs = [[rng.standard_normal((total, D)).astype(np.float16) for _ in range(Hkv)] for _ in lens]
    return Ks, Vs


@pytest.mark.parametrize("Hq,Hkv,G,Gv,R,bk,bv,lens", [
    (2, 2, 32, 32, 128, 2, 2, [1, 129, 700, 1537]),      # per-head kernel
    (8, 2, 32, 32, 128, 2, 2, [300, 1024, 2001]),        # grouped-query tensor-core kernel
    (4, 2, 64, 128, 128, 2, 2, [640, 999]),
    (2, 1, 32, 32, 256, 4, 4, [900, 1500]),              # 4-bit widths
    (3, 3, 128, 64, 128, 4, 2, [777, 256]),
])
def test_paged_decode_equals_dense_and_oracle(K, orc, Hq, Hkv, G, Gv, R, bk, bv, lens):
    rng = np.random.default_rng(sum(lens) + Hq + G + bk)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=G, group_v=Gv, residual=R, bits_k=bk, bits_v=bv)
    Ks, Vs = _data(rng, lens, Hkv)
    q = rng.standard_normal((len(lens), Hq, D)).astype(np.float16)
    max_seq_len = max(lens) + 3
    n_pages = sum((L + 127) // 128 for L in lens) + 7
    paged = _paged(cfg, Ks, Vs, lens, max_seq_len, n_pages, seed=5)
    dense = _dense(cfg, Ks, Vs, lens, max_seq_len)
    a = _decode(K, cfg, paged, q, True)
    assert torch.equal(a, _decode(K, cfg, dense, q, False))
    assert_attn_close(a.float().cpu().numpy(), _oracle(orc, cfg, Ks, Vs, q, lens))


def test_paged_append_matches_fill(K, orc):
    rng = np.random.default_rng(77)
    Hq, Hkv, G, R = 8, 2, 32, 128
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=G, residual=R)
    L0, n = [1, 250, 127], 300
    total = max(L0) + n
    Ks, Vs = _data(rng, L0, Hkv, total)
    n_pages = 40
    grown = _paged(cfg, Ks, Vs, L0, total + 5, n_pages, seed=9)
    top0 = int(grown.top[0].item())
    pool = grown.pool()
    for step in range(n):
        kn = torch.from_numpy(np.stack([np.stack([Ks[b][h][L0[b] + step] for h in range(Hkv)]) for b in range(3)]))
        vn = torch.from_numpy(np.stack([np.stack([Vs[b][h][L0[b] + step] for h in range(Hkv)]) for b in range(3)]))
        K.kv_append_kivi_paged(cfg, grown.desc(), pool, kn.to(DEV), vn.to(DEV))
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    lens = [L + n for L in L0]
    assert grown.seq_len.cpu().tolist() == lens
    used = sum((L + 127) // 128 for L in lens)
    assert top0 - int(grown.top[0].item()) == used - sum((L + 127) // 128 for L in L0)
    full = _paged(cfg, Ks, Vs, lens, total + 5, n_pages)
    # the quantized bytes of every logical page agree (physical pages differ)
    pb = grown.page_bytes
    kc, vc = 16 * D * 2, 16 * D * 2
    for b, L in enumerate(lens):
        nkq, nvq = kivi_segments(L, R)
        for j in range((L + 127) // 128):
            pg, pf = int(grown.page_table[b, j]), int(full.page_table[b, j])
            gk = max(0, min(128, nkq - 128 * j)) // G           # complete key groups in this page
            tv = max(0, min(128, nvq - 128 * j))                # quantized value tokens in this page
            for h in range(Hkv):
                x, y = grown.pages[pg, h], full.pages[pf, h]
                assert torch.equal(x[:gk * G * D // 4], y[:gk * G * D // 4])
                assert torch.equal(x[kc:kc + gk * 512], y[kc:kc + gk * 512])
                assert torch.equal(x[kc + 2048:kc + 2048 + tv * 32], y[kc + 2048:kc + 2048 + tv * 32])
                o = kc + 2048 + vc
                assert torch.equal(x[o:o + tv * 16], y[o:o + tv * 16])
        assert pb == kc + 2048 + vc + 2048
    q = rng.standard_normal((3, Hq, D)).astype(np.float16)
    a = _decode(K, cfg, grown, q, True)
    assert torch.equal(a, _decode(K, cfg, full, q, True))
    assert_attn_close(a.float().cpu().numpy(), _oracle(orc, cfg, Ks, Vs, q, lens))


def test_paged_pool_exhaustion_and_release(K):
    cfg = K.make_config(n_q_heads=2, n_kv_heads=1)
    rng = np.random.default_rng(13)
    lens = [256, 128, 1]
    Ks, Vs = _data(rng, lens, 1, 600)
    c = _paged(cfg, Ks, Vs, lens, 600, 4)                       # 2 + 1 + 1 pages: pool empty
    assert int(c.top[0].item()) == 0
    kn = torch.from_numpy(rng.standard_normal((3, 1, D)).astype(np.float16)).to(DEV)
    before = [t.clone() for t in (c.seq_len, c.pages, c.k_res)]
    K.kv_append_kivi_paged(cfg, c.desc(), c.pool(), kn, kn)    # rows 0 and 1 need a page, none is free
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_POOL
    assert c.seq_len.cpu().tolist() == [256, 128, 2]            # row 2 did not need a page
    assert torch.equal(c.k_res[:2], before[2][:2])
    rel = c.page_table[0, :2].clone()
    K.kv_release_kivi_paged(c.desc(), 0, c.pool())
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert int(c.top[0].item()) == 2 and torch.equal(c.free_pages[:2], rel)
    assert c.seq_len.cpu().tolist() == [0, 128, 2]
    K.kv_append_kivi_paged(cfg, c.desc(), c.pool(), kn, kn)    # rows 0 and 1 take the two released pages
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert c.seq_len.cpu().tolist() == [1, 129, 3] and int(c.top[0].item()) == 0


def test_paged_append_decode_graph_replay(K):
    cfg = K.make_config(n_q_heads=8, n_kv_heads=2)
    rng = np.random.default_rng(21)
    B, n = 2, 140
    lens = [200, 120]
    Ks, Vs = _data(rng, lens, 2, 400)
    eager = _paged(cfg, Ks, Vs, lens, 400, 16, seed=2)
    graphed = _paged(cfg, Ks, Vs, lens, 400, 16, seed=2)
    q = torch.from_numpy(rng.standard_normal((B, 8, D)).astype(np.float16)).to(DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI_PAGED, B, 400)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=DEV)
    out = torch.zeros((B, 8, D), dtype=torch.float16, device=DEV)
    kn = torch.zeros((B, 2, D), dtype=torch.float16, device=DEV)
    vn = torch.zeros_like(kn)
    desc, pool = graphed.desc(), graphed.pool()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        K.kv_append_kivi_paged(cfg, desc, pool, kn, vn, stream=torch.cuda.current_stream())
        K.kv_decode_attn_kivi_paged(cfg, desc, q, out, ws, wsb, stream=torch.cuda.current_stream())
    for step in range(n):
        kn.copy_(torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)))
        vn.copy_(torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)))
        graph.replay()
        g_out = out.clone()
        K.kv_append_kivi_paged(cfg, eager.desc(), eager.pool(), kn, vn)
        assert torch.equal(g_out, _decode(K, cfg, eager, q, True)), step
    assert K.kvq_get_device_error() == 0
    assert torch.equal(eager.page_table, graphed.page_table) and torch.equal(eager.pages, graphed.pages)
