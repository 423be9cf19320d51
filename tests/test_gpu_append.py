"""Streaming append (kv_append_kivi, kv_append_int8, kv_append_kitty): a cache grown token by token must
hold the bytes of a cache filled at once (the same quantizers; KIVI section
3.3 with the insert -> attend -> quantize order, Kitty "Stage 1" and "Stage 3" of its
pipeline, WitCert section 6.1 tail blocks),
and decode identically."""
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


def _segments(L, R):
    rk = (L - 1) % R + 1
    return L - rk, L - min(L, R)


def _fill(K, cfg, Ks, Vs, L_each, max_seq_len):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    c = C.KiviCache(cfg, B, max_seq_len, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            c.fill(b, h, Ks[b][h][:L_each[b]].to(DEV), Vs[b][h][:L_each[b]].to(DEV))
    return c


def _decode(K, cfg, c, q):
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, c.batch, c.max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((c.batch, cfg.n_q_heads, D), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn(cfg, c.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("Hq,Hkv,G,Gv,R,L0,n", [
    (4, 2, 32, 32, 128, 1, 300),       # from one token across three key flushes
    (2, 2, 64, 64, 128, 250, 200),
    (8, 2, 128, 128, 128, 127, 140),   # a flush on the first append
    (4, 4, 32, 32, 64, 500, 130),
])
def test_append_matches_fill(K, orc, Hq, Hkv, G, Gv, R, L0, n):
    rng = np.random.default_rng(L0 + n + G)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=G, group_v=Gv, residual=R)
    B = 2
    L_start = [L0, L0 + 7]
    total = max(L_start) + n
    max_seq_len = total + 3
    gain = 1.0 + 9.0 * (rng.random(D) < 0.05)
    Ks = [[torch.from_numpy((rng.standard_normal((total, D)) * gain).astype(np.float16)) for _ in range(Hkv)]
          for _ in range(B)]
    Vs = [[torch.from_numpy(rng.standard_normal((total, D)).astype(np.float16)) for _ in range(Hkv)] for _ in range(B)]
    grown = _fill(K, cfg, Ks, Vs, L_start, max_seq_len)
    for step in range(n):
        kn = torch.stack([torch.stack([Ks[b][h][L_start[b] + step] for h in range(Hkv)]) for b in range(B)]).to(DEV)
        vn = torch.stack([torch.stack([Vs[b][h][L_start[b] + step] for h in range(Hkv)]) for b in range(B)]).to(DEV)
        K.kv_append_kivi(cfg, grown.desc(), kn, vn)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    L_end = [L + n for L in L_start]
    full = _fill(K, cfg, Ks, Vs, L_end, max_seq_len)
    assert grown.seq_len.cpu().tolist() == L_end
    for b in range(B):
        nkq, nvq = _segments(L_end[b], R)
        ng = nkq // G
        assert torch.equal(grown.k_codes[b, :, :ng], full.k_codes[b, :, :ng])
        assert torch.equal(grown.k_sz[b, :, :ng], full.k_sz[b, :, :ng])
        assert torch.equal(grown.v_codes[b, :, :nvq], full.v_codes[b, :, :nvq])
        assert torch.equal(grown.v_sz[b, :, :nvq], full.v_sz[b, :, :nvq])
        kslots = [t % R for t in range(nkq, L_end[b])]
        vslots = [t % R for t in range(nvq, L_end[b])]
        assert torch.equal(grown.k_res[b, :, kslots], full.k_res[b, :, kslots])
        assert torch.equal(grown.v_res[b, :, vslots], full.v_res[b, :, vslots])
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float16)).to(DEV)
    a, f = _decode(K, cfg, grown, q), _decode(K, cfg, full, q)
    assert torch.equal(a, f)
    g = Hq // Hkv
    want = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hkv):
            parts = orc.kivi_build_one(Ks[b][h][:L_end[b]].numpy(), Vs[b][h][:L_end[b]].numpy(), G, Gv, R)
            want[b, h * g:(h + 1) * g] = orc.kivi_decode_one(q[b, h * g:(h + 1) * g].cpu().numpy(), *parts,
                                                             L=L_end[b], G=G, Gv=Gv, R=R)
    assert_attn_close(a.float().cpu().numpy(), want)


def test_append_full_row_reports_capacity(K):
    cfg = K.make_config(n_q_heads=2, n_kv_heads=2)
    rng = np.random.default_rng(3)
    Ks = [[torch.from_numpy(rng.standard_normal((256, D)).astype(np.float16)) for _ in range(2)]]
    Vs = [[torch.from_numpy(rng.standard_normal((256, D)).astype(np.float16)) for _ in range(2)]]
    c = _fill(K, cfg, Ks, Vs, [256], 256)
    before = (c.k_res.clone(), c.v_res.clone(), c.k_codes.clone(), c.v_codes.clone())
    kn = torch.zeros((1, 2, D), dtype=torch.float16, device=DEV)
    K.kv_append_kivi(cfg, c.desc(), kn, kn)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_CAPACITY
    assert K.kvq_get_device_error() == 0                      # reading clears it
    assert c.seq_len.cpu().tolist() == [256]
    after = (c.k_res, c.v_res, c.k_codes, c.v_codes)
    assert all(torch.equal(x, y) for x, y in zip(before, after))


def test_append_and_decode_in_one_graph(K):
    """Append + decode captured once and replayed step by step equals the eager loop."""
    cfg = K.make_config(n_q_heads=4, n_kv_heads=2)
    rng = np.random.default_rng(11)
    B, Hkv, n = 2, 2, 40
    total = 200 + n
    Ks = [[torch.from_numpy(rng.standard_normal((total, D)).astype(np.float16)) for _ in range(Hkv)]
          for _ in range(B)]
    Vs = [[torch.from_numpy(rng.standard_normal((total, D)).astype(np.float16)) for _ in range(Hkv)] for _ in range(B)]
    q = torch.from_numpy(rng.standard_normal((B, 4, D)).astype(np.float16)).to(DEV)
    eager = _fill(K, cfg, Ks, Vs, [200, 190], total)
    graphed = _fill(K, cfg, Ks, Vs, [200, 190], total)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, total)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=DEV)
    out = torch.zeros((B, 4, D), dtype=torch.float16, device=DEV)
    kn = torch.zeros((B, Hkv, D), dtype=torch.float16, device=DEV)
    vn = torch.zeros_like(kn)
    stream = torch.cuda.Stream()
    desc = graphed.desc()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        K.kv_append_kivi(cfg, desc, kn, vn, stream=torch.cuda.current_stream())
        K.kv_decode_attn(cfg, desc, q, out, ws, wsb, stream=torch.cuda.current_stream())
    outs_e, outs_g = [], []
    for step in range(n):
        cur = [200 + step, 190 + step]
        kn.copy_(torch.stack([torch.stack([Ks[b][h][cur[b]] for h in range(Hkv)]) for b in range(B)]))
        vn.copy_(torch.stack([torch.stack([Vs[b][h][cur[b]] for h in range(Hkv)]) for b in range(B)]))
        graph.replay()
        outs_g.append(out.clone())
        K.kv_append_kivi(cfg, eager.desc(), kn, vn)
        outs_e.append(_decode(K, cfg, eager, q))
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    for a, b in zip(outs_e, outs_g):
        assert torch.equal(a, b)


def _fill_int8(cfg, Ks, Vs, L_each, max_seq_len, reqs, layer, seed):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    c = C.Int8Cache(cfg, B, max_seq_len, layer=layer, seed=seed, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            c.fill(b, h, Ks[b][h][:L_each[b]].to(DEV), Vs[b][h][:L_each[b]].to(DEV), int(reqs[b]))
    return c


@pytest.mark.parametrize("Hq,Hkv,L0,n", [(8, 2, 1, 600), (4, 4, 255, 300), (8, 1, 700, 100)])
def test_append_int8_matches_fill(K, orc, Hq, Hkv, L0, n):
    rng = np.random.default_rng(L0 + n)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    B, T, layer, seed = 2, cfg.int8_block, 3, 0xABCDEF0123
    reqs = rng.integers(0, 2 ** 31 - 1, B)
    L_start = [L0, L0 + 31]
    total = max(L_start) + n
    max_seq_len = total + 5
    Ks = [[torch.from_numpy((rng.standard_normal((total, D)) * 10.0 ** rng.uniform(-1, 1, D)).astype(np.float16))
           for _ in range(Hkv)] for _ in range(B)]
    Vs = [[torch.from_numpy(rng.standard_normal((total, D)).astype(np.float16)) for _ in range(Hkv)] for _ in range(B)]
    grown = _fill_int8(cfg, Ks, Vs, L_start, max_seq_len, reqs, layer, seed)
    for step in range(n):
        kn = torch.stack([torch.stack([Ks[b][h][L_start[b] + step] for h in range(Hkv)]) for b in range(B)]).to(DEV)
        vn = torch.stack([torch.stack([Vs[b][h][L_start[b] + step] for h in range(Hkv)]) for b in range(B)]).to(DEV)
        K.kv_append_int8(cfg, grown.desc(), kn, vn)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    L_end = [L + n for L in L_start]
    full = _fill_int8(cfg, Ks, Vs, L_end, max_seq_len, reqs, layer, seed)
    assert grown.seq_len.cpu().tolist() == L_end
    for b in range(B):
        nq = L_end[b] - ((L_end[b] - 1) % T + 1)
        assert torch.equal(grown.k_codes[b, :, :nq], full.k_codes[b, :, :nq])
        assert torch.equal(grown.v_codes[b, :, :nq], full.v_codes[b, :, :nq])
        assert torch.equal(grown.k_scale[b, :, :nq // T], full.k_scale[b, :, :nq // T])
        assert torch.equal(grown.v_scale[b, :, :nq // T], full.v_scale[b, :, :nq // T])
        slots = [t % T for t in range(nq, L_end[b])]
        assert torch.equal(grown.k_tail[b, :, slots], full.k_tail[b, :, slots])
        assert torch.equal(grown.v_tail[b, :, slots], full.v_tail[b, :, slots])
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float16)).to(DEV)
    outs = []
    for c in (grown, full):
        _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8, B, max_seq_len)
        ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device=DEV)
        K.kv_decode_attn_int8(cfg, c.desc(), q, out, ws, wsb)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    g = Hq // Hkv
    want = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hkv):
            parts = orc.int8_build_one(Ks[b][h][:L_end[b]].numpy(), Vs[b][h][:L_end[b]].numpy(), seed, int(reqs[b]),
                                       layer, h)
            want[b, h * g:(h + 1) * g] = orc.int8_decode_one(q[b, h * g:(h + 1) * g].cpu().numpy(), *parts,
                                                             L=L_end[b], seed=seed, request=int(reqs[b]), layer=layer,
                                                             kv_head=h)
    assert_attn_close(outs[0].float().cpu().numpy(), want)


def _fill_kitty(cfg, Ks, Vs, L_each, max_seq_len, score_mode):
    from bit_kv_cache_keyquant_gb300 import cache as C
    B, Hkv = len(Ks), len(Ks[0])
    c = C.KittyCache(cfg, B, max_seq_len, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            c.fill(b, h, Ks[b][h][:L_each[b]].to(DEV), Vs[b][h][:L_each[b]].to(DEV), score_mode)
    return c


@pytest.mark.parametrize("Hq,Hkv,Kb,mode,L0,n", [
    (4, 2, 16, 0, 1, 450),      # sink, then two key-page and two value-page flushes
    (8, 2, 48, 1, 150, 300),
    (2, 1, 0, 0, 287, 140),     # a value-page flush on the first append
])
def test_append_kitty_matches_fill(K, orc, Hq, Hkv, Kb, mode, L0, n):
    from bit_kv_cache_keyquant_gb300.cache import kitty_segments
    rng = np.random.default_rng(L0 + n + Kb)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, group_k=128, boost_k=Kb)
    G, S, R = cfg.group_k, cfg.sink, cfg.residual
    B = 2
    L_start = [L0, L0 + 5]
    total = max(L_start) + n
    max_seq_len = total + 2
    gain = 1.0 + 9.0 * (rng.random(D) < 0.1)
    Ks = [[torch.from_numpy((rng.standard_normal((total, D)) * gain).astype(np.float16)) for _ in range(Hkv)]
          for _ in range(B)]
    Vs = [[torch.from_numpy(rng.standard_normal((total, D)).astype(np.float16)) for _ in range(Hkv)] for _ in range(B)]
    grown = _fill_kitty(cfg, Ks, Vs, L_start, max_seq_len, mode)
    for step in range(n):
        kn = torch.stack([torch.stack([Ks[b][h][L_start[b] + step] for h in range(Hkv)]) for b in range(B)]).to(DEV)
        vn = torch.stack([torch.stack([Vs[b][h][L_start[b] + step] for h in range(Hkv)]) for b in range(B)]).to(DEV)
        K.kv_append_kitty(cfg, grown.desc(), kn, vn, mode)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    L_end = [L + n for L in L_start]
    full = _fill_kitty(cfg, Ks, Vs, L_end, max_seq_len, mode)
    assert grown.seq_len.cpu().tolist() == L_end
    for b in range(B):
        L = L_end[b]
        pk, nkb, pv, nvb, nloc = kitty_segments(L, G, S, R)
        ns = min(L, S)
        assert torch.equal(grown.k_pages[b, :, :pk], full.k_pages[b, :, :pk])
        assert torch.equal(grown.v_pages[b, :, :pv], full.v_pages[b, :, :pv])
        assert torch.equal(grown.k_sink[b, :, :ns], full.k_sink[b, :, :ns])
        assert torch.equal(grown.v_sink[b, :, :ns], full.v_sink[b, :, :ns])
        k0, v0 = S + pk * G, S + pv * G
        kslots = [(t - S) % G for t in range(k0, L)]
        vslots = [(t - S) % G for t in range(v0, v0 + nvb)]
        lslots = [t % R for t in range(L - nloc, L)]
        assert torch.equal(grown.k_qbuf[b, :, kslots], full.k_qbuf[b, :, kslots])
        assert torch.equal(grown.v_qbuf[b, :, vslots], full.v_qbuf[b, :, vslots])
        assert torch.equal(grown.v_local[b, :, lslots], full.v_local[b, :, lslots])
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float16)).to(DEV)
    outs = []
    for c in (grown, full):
        _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KITTY, B, max_seq_len)
        ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float16, device=DEV)
        K.kv_decode_attn_kitty(cfg, c.desc(), q, out, ws, wsb)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])
    g = Hq // Hkv
    want = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hkv):
            parts = orc.kitty_build_one(Ks[b][h][:L_end[b]].numpy(), Vs[b][h][:L_end[b]].numpy(), G, Kb, S, R, mode)
            want[b, h * g:(h + 1) * g] = orc.kitty_decode_one(q[b, h * g:(h + 1) * g].cpu().numpy(), *parts,
                                                              L=L_end[b], K=Kb, S=S, R=R)
    assert_attn_close(outs[0].float().cpu().numpy(), want)


def test_append_kitty_full_row_reports_capacity(K):
    cfg = K.make_config(n_q_heads=2, n_kv_heads=1, group_k=128)
    rng = np.random.default_rng(5)
    L = 300
    Ks = [[torch.from_numpy(rng.standard_normal((L, D)).astype(np.float16))]]
    Vs = [[torch.from_numpy(rng.standard_normal((L, D)).astype(np.float16))]]
    c = _fill_kitty(cfg, Ks, Vs, [L], L, 0)
    before = [t.clone() for t in (c.k_pages, c.v_pages, c.k_qbuf, c.v_qbuf, c.v_local, c.k_sink)]
    kn = torch.zeros((1, 1, D), dtype=torch.float16, device=DEV)
    K.kv_append_kitty(cfg, c.desc(), kn, kn, 0)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_CAPACITY
    assert c.seq_len.cpu().tolist() == [L]
    after = (c.k_pages, c.v_pages, c.k_qbuf, c.v_qbuf, c.v_local, c.k_sink)
    assert all(torch.equal(x, y) for x, y in zip(before, after))
