"""GPU parity of the token-granular INT8 slot-pool path (WitCert, SGLang storage subsection of
sec. 6.2): per-token Gc-channel scales, dither keyed by slot, decode through a per-request slot
table, and the device free-slot stack of the streaming append."""
import numpy as np
import pytest
import torch

from bit_kv_cache_keyquant_gb300 import inputs as I
from tests.gpu_util import assert_attn_close, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128


@pytest.fixture(scope="module")
def K():
    return lib()


def _cache(K, cfg, B, max_seq_len, n_slots, layer, seed, shuffle_seed=None):
    from bit_kv_cache_keyquant_gb300 import cache as C
    c = C.Int8TokenCache(cfg, B, max_seq_len, n_slots, layer=layer, seed=seed, device=DEV)
    if shuffle_seed is not None:
        rng = np.random.default_rng(shuffle_seed)
        c.shuffle_free(rng.permutation(n_slots // 16), 16)
    return c


def _pool_np(c):
    return (c.k_codes.cpu().numpy(), c.v_codes.cpu().numpy(), c.k_scale.cpu().numpy().view(np.uint16),
            c.v_scale.cpu().numpy().view(np.uint16))


def _decode(K, cfg, c, q):
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8_TOKEN, c.batch, c.max_seq_len)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((c.batch, cfg.n_q_heads, D), float("nan"), dtype=torch.float16, device=DEV)
    K.kv_decode_attn_int8_token(cfg, c.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    return out


def _oracle(orc, cfg, c, q, lens):
    pool = _pool_np(c)
    table = c.slot_table.cpu().numpy()
    g = cfg.n_q_heads // cfg.n_kv_heads
    qn = q.cpu().numpy()
    want = np.zeros((c.batch, cfg.n_q_heads, D))
    for b, L in enumerate(lens):
        for h in range(cfg.n_kv_heads):
            if L == 0:
                continue
            want[b, h * g:(h + 1) * g] = orc.int8t_decode_one(qn[b, h * g:(h + 1) * g], pool, table[b, :L], h,
                                                              c.seed, c.layer, cfg.int8_group)
    return want


@pytest.mark.parametrize("Gc", [32, 64, 128])
def test_quant_token_matches_oracle(K, orc, Gc):
    rng = np.random.default_rng(Gc)
    Hkv, n, n_slots = 3, 70, 500
    cfg = K.make_config(n_q_heads=6, n_kv_heads=Hkv, int8_group=Gc)
    c = _cache(K, cfg, 1, 8, n_slots, layer=9, seed=0x123456789ABCDEF)
    x = (rng.standard_normal((n, Hkv, D)) * 10.0 ** rng.uniform(-3, 3, (n, Hkv, D))).astype(np.float16)
    x[0, 1] = 0                                           # an all-zero token: s = 0, codes 0
    x[1, 2, :Gc] = np.float16(60000)                      # near the fp16 maximum
    slots = rng.permutation(n_slots)[:n].astype(np.int32)
    slots[5] = -1                                         # outside the pool: skipped
    xt = torch.from_numpy(x).to(DEV)
    st = torch.from_numpy(slots).to(DEV)
    K.kv_quant_int8_token(cfg, c.desc(), xt, n, st, 0)
    K.kv_quant_int8_token(cfg, c.desc(), xt, n, st, 1)
    torch.cuda.synchronize()
    kc, vc, ks, vs = _pool_np(c)
    for i in range(n):
        if slots[i] < 0:
            continue
        for h in range(Hkv):
            for sel, (cc, ss) in enumerate(((kc, ks), (vc, vs))):
                codes, scale = orc.int8t_quant_token(x[i, h], Gc, c.seed, 9, sel, h, int(slots[i]))
                assert np.array_equal(cc[slots[i], h], codes), (i, h, sel)
                assert np.array_equal(ss[slots[i], h], scale), (i, h, sel)
    untouched = np.setdiff1d(np.arange(n_slots), slots)
    assert not kc[untouched].any() and not ks[untouched].any()


@pytest.mark.parametrize("Hq,Hkv,Gc,lens", [
    (8, 1, 32, [1, 100, 129]),
    (16, 2, 32, [700, 0, 1500]),          # an empty request gives 0
    (6, 3, 64, [257, 1024]),
    (8, 8, 128, [300, 33]),
    (64, 8, 32, [2000, 1111]),
])
def test_decode_parity(K, orc, Hq, Hkv, Gc, lens):
    rng = np.random.default_rng(sum(lens) + Hq + Gc)
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv, int8_group=Gc)
    n_slots = (sum(lens) + 64) // 16 * 16 + 64
    c = _cache(K, cfg, len(lens), max(lens) + 3, n_slots, layer=3, seed=0xABCDEF, shuffle_seed=7)
    for b, L in enumerate(lens):
        if L:
            Kt = (rng.standard_normal((L, Hkv, D)) * 10.0 ** rng.uniform(-1, 1, (1, Hkv, D))).astype(np.float16)
            Vt = rng.standard_normal((L, Hkv, D)).astype(np.float16)
            c.fill(b, torch.from_numpy(Kt).to(DEV), torch.from_numpy(Vt).to(DEV))
    q = torch.from_numpy(rng.standard_normal((len(lens), Hq, D)).astype(np.float16)).to(DEV)
    out = _decode(K, cfg, c, q)
    assert K.kvq_get_device_error() == 0
    got = out.float().cpu().numpy()
    assert_attn_close(got, _oracle(orc, cfg, c, q, lens))
    for b, L in enumerate(lens):
        if L == 0:
            assert not got[b].any()


def test_append_allocates_deterministically_and_matches_oracle(K, orc):
    rng = np.random.default_rng(31)
    Hq, Hkv, B, n = 8, 2, 3, 150
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    L0 = [5, 0, 300]
    n_slots = 1024
    c = _cache(K, cfg, B, 600, n_slots, layer=1, seed=99, shuffle_seed=3)
    Ks = [rng.standard_normal((L0[b] + n, Hkv, D)).astype(np.float16) for b in range(B)]
    Vs = [rng.standard_normal((L0[b] + n, Hkv, D)).astype(np.float16) for b in range(B)]
    for b in range(B):
        if L0[b]:
            c.fill(b, torch.from_numpy(Ks[b][:L0[b]]).to(DEV), torch.from_numpy(Vs[b][:L0[b]]).to(DEV))
    top0 = int(c.top[0].item())
    free0 = c.free_slots[:top0].cpu().numpy()
    pool = c.pool()
    for step in range(n):
        kn = torch.from_numpy(np.stack([Ks[b][L0[b] + step] for b in range(B)])).to(DEV)
        vn = torch.from_numpy(np.stack([Vs[b][L0[b] + step] for b in range(B)])).to(DEV)
        K.kv_append_int8_token(cfg, c.desc(), pool, kn, vn)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    lens = [L0[b] + n for b in range(B)]
    assert c.seq_len.cpu().tolist() == lens
    assert int(c.top[0].item()) == top0 - B * n
    table = c.slot_table.cpu().numpy()
    # step s, row b takes the (B*s + b)-th slot from the top of the stack
    for step in range(n):
        for b in range(B):
            assert table[b, L0[b] + step] == free0[top0 - 1 - (B * step + b)]
    # every appended token's codes equal the oracle's for its slot
    kc, vc, ks, vs = _pool_np(c)
    for b in range(B):
        for t in range(L0[b], lens[b], 37):
            s_ = int(table[b, t])
            for h in range(Hkv):
                codes, scale = orc.int8t_quant_token(Ks[b][t, h], 32, 99, 1, 0, h, s_)
                assert np.array_equal(kc[s_, h], codes) and np.array_equal(ks[s_, h], scale)
                codes, scale = orc.int8t_quant_token(Vs[b][t, h], 32, 99, 1, 1, h, s_)
                assert np.array_equal(vc[s_, h], codes) and np.array_equal(vs[s_, h], scale)
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float16)).to(DEV)
    assert_attn_close(_decode(K, cfg, c, q).float().cpu().numpy(), _oracle(orc, cfg, c, q, lens))


def test_pool_exhaustion_and_release(K):
    cfg = K.make_config(n_q_heads=4, n_kv_heads=2)
    B = 3
    c = _cache(K, cfg, B, 64, 40, layer=0, seed=5)
    rng = np.random.default_rng(8)
    c.fill(0, torch.from_numpy(rng.standard_normal((20, 2, D)).astype(np.float16)).to(DEV),
           torch.from_numpy(rng.standard_normal((20, 2, D)).astype(np.float16)).to(DEV))
    c.fill(1, torch.from_numpy(rng.standard_normal((18, 2, D)).astype(np.float16)).to(DEV),
           torch.from_numpy(rng.standard_normal((18, 2, D)).astype(np.float16)).to(DEV))
    assert int(c.top[0].item()) == 2
    kn = torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)).to(DEV)
    before = [t.clone() for t in (c.seq_len, c.k_codes, c.v_codes, c.free_slots, c.top)]
    K.kv_append_int8_token(cfg, c.desc(), c.pool(), kn, kn)          # 3 rows, 2 free slots
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_POOL
    after = (c.seq_len, c.k_codes, c.v_codes, c.free_slots, c.top)
    assert all(torch.equal(x, y) for x, y in zip(before, after))
    # releasing request 0 returns its 20 slots; the append then succeeds
    slots0 = c.slot_table[0, :20].clone()
    K.kv_release_int8_token(c.desc(), 0, c.pool())
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert c.seq_len.cpu().tolist() == [0, 18, 0]
    assert int(c.top[0].item()) == 22
    assert torch.equal(c.free_slots[2:22], slots0)
    K.kv_append_int8_token(cfg, c.desc(), c.pool(), kn, kn)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert c.seq_len.cpu().tolist() == [1, 19, 1]
    assert int(c.top[0].item()) == 19
    # a row at capacity is flagged and left alone
    c2 = _cache(K, cfg, 1, 4, 16, layer=0, seed=5)
    c2.fill(0, kn[:1].expand(4, 2, D).contiguous(), kn[:1].expand(4, 2, D).contiguous())
    K.kv_append_int8_token(cfg, c2.desc(), c2.pool(), kn[:1].contiguous(), kn[:1].contiguous())
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == K.KVQ_DEVICE_ERR_CAPACITY
    assert c2.seq_len.cpu().tolist() == [4] and int(c2.top[0].item()) == 12


def test_append_decode_graph_replay_is_bit_identical(K):
    """Append + decode captured once and replayed equals the eager loop bit for bit: the slots come
    from the free stack in a fixed order, so the dither of every written token is the same."""
    cfg = K.make_config(n_q_heads=16, n_kv_heads=2)
    rng = np.random.default_rng(12)
    B, n = 2, 30
    eager = _cache(K, cfg, B, 400, 1024, layer=2, seed=17, shuffle_seed=1)
    graphed = _cache(K, cfg, B, 400, 1024, layer=2, seed=17, shuffle_seed=1)
    K0 = rng.standard_normal((200, 2, D)).astype(np.float16)
    V0 = rng.standard_normal((200, 2, D)).astype(np.float16)
    for c in (eager, graphed):
        c.fill(0, torch.from_numpy(K0).to(DEV), torch.from_numpy(V0).to(DEV))
        c.fill(1, torch.from_numpy(K0[:150]).to(DEV), torch.from_numpy(V0[:150]).to(DEV))
    q = torch.from_numpy(rng.standard_normal((B, 16, D)).astype(np.float16)).to(DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_INT8_TOKEN, B, 400)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=DEV)
    out = torch.zeros((B, 16, D), dtype=torch.float16, device=DEV)
    kn = torch.zeros((B, 2, D), dtype=torch.float16, device=DEV)
    vn = torch.zeros_like(kn)
    desc, pool = graphed.desc(), graphed.pool()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):
        K.kv_append_int8_token(cfg, desc, pool, kn, vn, stream=torch.cuda.current_stream())
        K.kv_decode_attn_int8_token(cfg, desc, q, out, ws, wsb, stream=torch.cuda.current_stream())
    for step in range(n):
        kn.copy_(torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)))
        vn.copy_(torch.from_numpy(rng.standard_normal((B, 2, D)).astype(np.float16)))
        graph.replay()
        g_out = out.clone()
        K.kv_append_int8_token(cfg, eager.desc(), eager.pool(), kn, vn)
        e_out = _decode(K, cfg, eager, q)
        assert torch.equal(g_out, e_out), step
    assert K.kvq_get_device_error() == 0
    assert torch.equal(eager.slot_table, graphed.slot_table)
    assert torch.equal(eager.k_codes, graphed.k_codes) and torch.equal(eager.v_scale, graphed.v_scale)


@pytest.mark.slow
def test_workload_full_size_sampled(K, orc):
    """The token-granular workload at full size (B8, 64q/8kv, lengths 16K-64K, scattered 16-slot pages):
    sampled (batch row, kv head) pairs against the oracle."""
    w = I.WORKLOADS[6]
    lens = I.seq_lens(w)
    cfg = K.make_config(n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads)
    n_slots = (int(lens.sum()) + 15) // 16 * 16 + 256
    from bit_kv_cache_keyquant_gb300 import cache as C
    c = C.Int8TokenCache(cfg, w.batch, int(lens.max()), n_slots, layer=5, seed=w.seed, device=DEV)
    c.shuffle_free(I.page_permutation(w, n_slots // 16), 16)
    for b in range(w.batch):
        L = int(lens[b])
        Kt = torch.stack([I.gen_kv_torch(w, I.T_K, b, h, L, DEV) for h in range(w.n_kv_heads)], dim=1)
        Vt = torch.stack([I.gen_kv_torch(w, I.T_V, b, h, L, DEV) for h in range(w.n_kv_heads)], dim=1)
        c.fill(b, Kt, Vt)
    q = I.gen_q_torch(w, DEV)
    out = _decode(K, cfg, c, q).float().cpu().numpy()
    assert K.kvq_get_device_error() == 0
    pool = _pool_np(c)
    table = c.slot_table.cpu().numpy()
    qn = q.cpu().numpy()
    g = w.n_q_heads // w.n_kv_heads
    for b, h in ((0, 0), (w.batch - 1, w.n_kv_heads - 1), (3, 5)):
        L = int(lens[b])
        want = orc.int8t_decode_one(qn[b, h * g:(h + 1) * g], pool, table[b, :L], h, c.seed, c.layer, 32)
        assert_attn_close(out[b, h * g:(h + 1) * g], want, f"row {b} kv head {h}")
