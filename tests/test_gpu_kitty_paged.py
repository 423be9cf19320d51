"""GPU parity of the paged Kitty cache: key and value page records from shared pools through a
per-request page table (logical page j holds tokens S + 128 j ..).  The same tokens decode bit-identically
from the per-request and the paged cache, match the oracle, and grow by streaming append into pages
taken from the free stack."""
import numpy as np
import pytest
import torch

from bit_kv_cache_keyquant_gb300.cache import kitty_segments
from tests.gpu_util import assert_attn_close, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.fixture(scope="module")
def K():
    return lib()


def _pages_needed(L, S):
    return (max(L - S, 0) + 127) // 128


def _paged(cfg, Ks, Vs, lens, max_seq_len, n_pages, mode=0, seed=None):
    from bit_kv_cache_keyquant_gb300 import cache as C
    c = C.KittyPagedCache(cfg, len(lens), max_seq_len, n_pages, device=DEV)
    if seed is not None:
        c.shuffle_free(np.random.default_rng(seed).permutation(n_pages))
    for b, L in enumerate(lens):
        c.fill(b, torch.from_numpy(np.stack([k[:L] for k in Ks[b]])).to(DEV),
               torch.from_numpy(np.stack([v[:L] for v in Vs[b]])).to(DEV), mode)
    return c


def _dense(cfg, Ks, Vs, lens, max_seq_len, mode=0):
    from bit_kv_cache_keyquant_gb300 import cache as C
    c = C.KittyCache(cfg, len(lens), max_seq_len, device=DEV)
    for b, L in enumerate(lens):
        for h in range(cfg.n_kv_heads):
            c.fill(b, h, torch.from_numpy(Ks[b][h][:L]).to(DEV), torch.from_numpy(Vs[b][h][:L]).to(DEV), mode)
    return c


def _decode(K, cfg, c, q):
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KITTY, c.batch, c.max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((c.batch, cfg.n_q_heads, D), float("nan"), dtype=torch.float16, device=DEV)
    qd = torch.from_numpy(q).to(DEV) if isinstance(q, np.ndarray) else q
    K.kv_decode_attn_kitty(cfg, c.desc(), qd, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    return out


def _oracle(orc, cfg, Ks, Vs, q, lens, mode=0):
    g = cfg.n_q_heads // cfg.n_kv_heads
    out = np.zeros((len(lens), cfg.n_q_heads, D))
    for b, L in enumerate(lens):
        for h in range(cfg.n_kv_heads):
            parts = orc.kitty_build_one(Ks[b][h][:L], Vs[b][h][:L], 128, cfg.boost_k, cfg.sink, cfg.residual, mode)
            out[b, h * g:(h + 1) * g] = orc.kitty_decode_one(q[b, h * g:(h + 1) * g], *parts, L=L, K=cfg.boost_k,
                                                             S=cfg.sink, R=cfg.residual)
    return out


def _data(rng, n_rows, Hkv, total):
    sig = 0.5 * 16.0 ** rng.random(D)
    Ks = [[(rng.standard_normal((total, D)) * sig).astype(np.float16) for _ in range(Hkv)] for _ in range(n_rows)]
    Vs = [[rng.standard_normal((total, D)).astype(np.float16) for _ in range(Hkv)] for _ in range(n_rows)]
    return Ks, Vs


@pytest.mark.parametrize("Hq,Hkv,Kb,mode,lens", [
    (2, 2, 16, 0, [1, 33, 200, 700]),          # per-head kernel; a row shorter than the sink
    (8, 2, 16, 1, [160, 1100, 2000]),          # grouped-query tensor-core kernel
    (4, 4, 32, 0, [417, 1500]),                # alpha = 0.25
    (1, 1, 0, 0, [900]),
])
def test_paged_kitty_equals_dense_and_oracle(K, orc, Hq, Hkv, Kb, mode, lens):
    rng = np.random.default_rng(sum(lens) + Hq + Kb)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, boost_k=Kb)
    Ks, Vs = _data(rng, len(lens), Hkv, max(lens))
    q = rng.standard_normal((len(lens), Hq, D)).astype(np.float16)
    max_seq_len = max(lens) + 3
    n_pages = sum(_pages_needed(L, cfg.sink) for L in lens) + 5
    paged = _paged(cfg, Ks, Vs, lens, max_seq_len, n_pages, mode, seed=4)
    dense = _dense(cfg, Ks, Vs, lens, max_seq_len, mode)
    a = _decode(K, cfg, paged, q)
    assert torch.equal(a, _decode(K, cfg, dense, q))
    assert_attn_close(a.float().cpu().numpy(), _oracle(orc, cfg, Ks, Vs, q, lens, mode))


def test_paged_kitty_append_matches_fill(K, orc):
    rng = np.random.default_rng(31)
    Hq, Hkv = 8, 2
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, boost_k=16)
    S, R = cfg.sink, cfg.residual
    L0, n = [1, 160, 290], 420
    total = max(L0) + n
    Ks, Vs = _data(rng, 3, Hkv, total)
    n_pages = 30
    grown = _paged(cfg, Ks, Vs, L0, total + 3, n_pages, seed=6)
    pool = grown.pool()
    for step in range(n):
        kn = torch.from_numpy(np.stack([np.stack([Ks[b][h][L0[b] + step] for h in range(Hkv)]) for b in range(3)]))
        vn = torch.from_numpy(np.stack([np.stack([Vs[b][h][L0[b] + step] for h in range(Hkv)]) for b in range(3)]))
        K.kv_append_kitty_paged(cfg, grown.desc(), pool, kn.to(DEV), vn.to(DEV))
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    lens = [L + n for L in L0]
    assert grown.seq_len.cpu().tolist() == lens
    assert n_pages - int(grown.top[0].item()) == sum(_pages_needed(L, S) for L in lens)
    full = _paged(cfg, Ks, Vs, lens, total + 3, n_pages)
    for b, L in enumerate(lens):
        pk, nkb, pv, nvb, nloc = kitty_segments(L, 128, S, R)
        for j in range(pk):
            x, y = int(grown.page_table[b, j]), int(full.page_table[b, j])
            assert torch.equal(grown.k_pages[x], full.k_pages[y])
        for j in range(pv):
            x, y = int(grown.page_table[b, j]), int(full.page_table[b, j])
            assert torch.equal(grown.v_pages[x], full.v_pages[y])
    q = rng.standard_normal((3, Hq, D)).astype(np.float16)
    a = _decode(K, cfg, grown, q)
    assert torch.equal(a, _decode(K, cfg, full, q))
    assert_attn_close(a.float().cpu().numpy(), _oracle(orc, cfg, Ks, Vs, q, lens))


def test_paged_kitty_pool_exhaustion_and_release(K):
    cfg = K.make_config(n_q_heads=2, n_kv_heads=1, group_k=128, boost_k=16)
    S = cfg.sink
    rng = np.random.default_rng(17)
    lens = [S + 256, S + 128, 5]                     # 2 + 1 + 0 pages
    Ks, Vs = _data(rng, 3, 1, 600)
    c = _paged(cfg, Ks, Vs, lens, 600, 3)
    assert int(c.top[0].item()) == 0
    kn = torch.from_numpy(rng.standard_normal((3, 1, D)).astype(np.float16)).to(DEV)
    before = (c.seq_len.clone(), c.k_pages.clone(), c.v_pages.clone(), c.k_qbuf.clone())
    K.kv_append_kitty_paged(cfg, c.desc(), c.pool(), kn, kn)   # rows 0 and 1 need a page, none is free
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_POOL
    assert c.seq_len.cpu().tolist() == [S + 256, S + 128, 6]
    assert torch.equal(c.k_pages, before[1]) and torch.equal(c.k_qbuf[:2], before[3][:2])
    rel = c.page_table[0, :2].clone()
    K.kv_release_kitty(cfg, c.desc(), 0, c.pool())
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert int(c.top[0].item()) == 2 and torch.equal(c.free_pages[:2], rel)
    assert c.seq_len.cpu().tolist() == [0, S + 128, 6]
    K.kv_append_kitty_paged(cfg, c.desc(), c.pool(), kn, kn)   # row 1 takes a page; row 0 restarts in the sink
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert c.seq_len.cpu().tolist() == [1, S + 129, 7] and int(c.top[0].item()) == 1


def test_paged_kitty_graph_replay(K):
    cfg = K.make_config(n_q_heads=8, n_kv_heads=2, group_k=128, boost_k=16)
    rng = np.random.default_rng(23)
    B, n = 2, 150
    lens = [150, 260]
    Ks, Vs = _data(rng, 2, 2, 600)
    eager = _paged(cfg, Ks, Vs, lens, 600, 12, seed=3)
    graphed = _paged(cfg, Ks, Vs, lens, 600, 12, seed=3)
    q = torch.from_numpy(rng.standard_normal((B, 8, D)).astype(np.float16)).to(DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KITTY, B, 600)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=DEV)
    out = torch.zeros((B, 8, D), dtype=torch.float16, device=DEV)
    kn = torch.zeros((B, 2, D), dtype=torch.float16, device=DEV)
    vn = torch.zeros_like(kn)
    desc, pool = graphed.desc(), graphed.pool()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        K.kv_append_kitty_paged(cfg, desc, pool, kn, vn, stream=torch.cuda.current_stream())
        K.kv_decode_attn_kitty(cfg, desc, q, out, ws, wsb, stream=torch.cuda.current_stream())
    for step in range(n):
        kn.copy_(torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)))
        vn.copy_(torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)))
        graph.replay()
        g_out = out.clone()
        K.kv_append_kitty_paged(cfg, eager.desc(), eager.pool(), kn, vn)
        assert torch.equal(g_out, _decode(K, cfg, eager, q)), step
    assert K.kvq_get_device_error() == 0
    assert torch.equal(eager.page_table, graphed.page_table) and torch.equal(eager.k_pages, graphed.k_pages)
