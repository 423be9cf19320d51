"""Device-resident KV caches in the layouts of include/kvq.h.

Each class owns the torch tensors of one cache (all batch rows and kv heads
of one layer), fills a (batch row, kv head) slice from fp16 keys and values
through the library's quantization entry points, and exposes the C
descriptor the decode entry points take.  Segment bookkeeping follows the
rules stated in include/kvq.h (Kitty's insert -> attend -> quantize order).
"""
from __future__ import annotations

import torch

from . import kvq

D = 128


def kivi_segments(L: int, R: int):
    """(quantized keys, quantized values) at attention time with L tokens."""
    rk = ((L - 1) % R) + 1
    return L - rk, L - min(L, R)


def kitty_segments(L: int, G: int, S: int, R: int):
    """(key pages, key Q-buffer, value pages, value Q-buffer, local window)."""
    if L > S:
        nkb = ((L - S - 1) % G) + 1
        pk = (L - S - nkb) // G
    else:
        nkb, pk = 0, 0
    E = max(0, L - S - R)
    nvb = ((E - 1) % G) + 1 if E > 0 else 0
    pv = (E - nvb) // G
    nloc = min(max(L - S, 0), R)
    return pk, nkb, pv, nvb, nloc


def int8_segments(L: int, T: int):
    """(quantized blocks, fp16 tail tokens)."""
    ntail = ((L - 1) % T) + 1
    return (L - ntail) // T, ntail


def _slot_copy(dst, src, slots):
    idx = torch.as_tensor(slots, dtype=torch.int64, device=dst.device)
    dst.index_copy_(0, idx, src)


class KiviCache:
    def __init__(self, cfg: kvq.kvq_config, batch: int, max_seq_len: int, device="cuda"):
        self.cfg, self.batch, self.max_seq_len = cfg, batch, max_seq_len
        H, G, Gv, R = cfg.n_kv_heads, cfg.group_k, cfg.group_v, cfg.residual
        self.cap = (max_seq_len + 127) // 128 * 128        # token capacity (16-byte aligned rows)
        self.ngrp_cap = self.cap // G
        bk, bv = cfg.bits_k, cfg.bits_v
        self.k_codes = torch.zeros((batch, H, self.ngrp_cap, G * D * bk // 8), dtype=torch.uint8, device=device)
        self.k_sz = torch.zeros((batch, H, self.ngrp_cap, D), dtype=torch.int32, device=device)
        self.v_codes = torch.zeros((batch, H, self.cap, D * bv // 8), dtype=torch.uint8, device=device)
        self.v_sz = torch.zeros((batch, H, self.cap, D // Gv), dtype=torch.int32, device=device)
        self.k_res = torch.zeros((batch, H, R, D), dtype=torch.float16, device=device)
        self.v_res = torch.zeros((batch, H, R, D), dtype=torch.float16, device=device)
        self.seq_len = torch.ones(batch, dtype=torch.int32, device=device)

    def fill(self, b: int, kvh: int, K: torch.Tensor, V: torch.Tensor, stream=None):
        """Quantize one (batch row, kv head) from fp16 K, V [L][D] on the device."""
        cfg = self.cfg
        L = K.shape[0]
        assert 1 <= L <= self.max_seq_len and K.shape == V.shape == (L, D)
        G, R = cfg.group_k, cfg.residual
        nkq, nvq = kivi_segments(L, R)
        if nkq:
            kvq.kv_quant_key(cfg, K[:nkq].contiguous(), nkq // G, self.k_codes[b, kvh], self.k_sz[b, kvh], stream)
        if nvq:
            kvq.kv_quant_value(cfg, V[:nvq].contiguous(), nvq, self.v_codes[b, kvh], self.v_sz[b, kvh], stream)
        _slot_copy(self.k_res[b, kvh], K[nkq:L], [t % R for t in range(nkq, L)])
        _slot_copy(self.v_res[b, kvh], V[nvq:L], [t % R for t in range(nvq, L)])
        self.seq_len[b] = L

    def desc(self) -> kvq.kvq_kivi_cache:
        return kvq.kvq_kivi_cache(self.batch, self.max_seq_len, self.seq_len.data_ptr(), self.k_codes.data_ptr(),
                                  self.k_sz.data_ptr(), self.v_codes.data_ptr(), self.v_sz.data_ptr(),
                                  self.k_res.data_ptr(), self.v_res.data_ptr())

    def nbytes_read(self, lens) -> int:
        """Algorithmic bytes one decode step reads from this cache (codes, (s, z), fp16 residual)."""
        cfg = self.cfg
        tot = 0
        for L in lens:
            nkq, nvq = kivi_segments(int(L), cfg.residual)
            tot += nkq * D * cfg.bits_k // 8 + (nkq // cfg.group_k) * D * 4     # key codes + (s, z)
            tot += nvq * D * cfg.bits_v // 8 + nvq * (D // cfg.group_v) * 4     # value codes + (s, z)
            tot += (int(L) - nkq + int(L) - nvq) * D * 2                 # fp16 residual
        return tot * cfg.n_kv_heads


class KiviPagedCache:
    """Paged KIVI cache of one layer: n_pages page records of 128 tokens x Hkv heads shared by all
    requests, a page table per request, a free-page stack, and per-(row, kv head) fp16 residual rings."""

    def __init__(self, cfg: kvq.kvq_config, batch: int, max_seq_len: int, n_pages: int, device="cuda"):
        self.cfg, self.batch, self.max_seq_len, self.n_pages = cfg, batch, max_seq_len, n_pages
        H, R = cfg.n_kv_heads, cfg.residual
        self.page_bytes = kvq.kvq_kivi_page_bytes(cfg)
        self.pt_stride = (max_seq_len + 127) // 128
        self.pages = torch.zeros((n_pages, H, self.page_bytes), dtype=torch.uint8, device=device)
        self.page_table = torch.full((batch, self.pt_stride), -1, dtype=torch.int32, device=device)
        self.seq_len = torch.zeros(batch, dtype=torch.int32, device=device)
        self.k_res = torch.zeros((batch, H, R, D), dtype=torch.float16, device=device)
        self.v_res = torch.zeros((batch, H, R, D), dtype=torch.float16, device=device)
        self.free_pages = torch.empty(n_pages, dtype=torch.int32, device=device)
        self.top = torch.zeros(4, dtype=torch.int32, device=device)
        kvq.kv_slot_pool_init(self.pool())

    def pool(self) -> kvq.kvq_slot_pool:
        return kvq.kvq_slot_pool(self.n_pages, self.free_pages.data_ptr(), self.top.data_ptr())

    def desc(self) -> kvq.kvq_kivi_paged_cache:
        return kvq.kvq_kivi_paged_cache(self.batch, self.max_seq_len, self.seq_len.data_ptr(),
                                        self.page_table.data_ptr(), self.n_pages, self.pages.data_ptr(),
                                        self.k_res.data_ptr(), self.v_res.data_ptr())

    def shuffle_free(self, perm):
        """Reorder the free stack by a permutation of its entries (host setup), so that later pops hand
        out scattered pages."""
        top = int(self.top[0].item())
        free = self.free_pages[:top].flip(0)
        idx = torch.as_tensor(perm, dtype=torch.int64, device=free.device)
        self.free_pages[:top] = free[idx].flip(0)

    def fill(self, b: int, K: torch.Tensor, V: torch.Tensor, stream=None):
        """Request b from fp16 K, V [Hkv][L][D]: pops ceil(L/128) pages, quantizes every head into them."""
        cfg = self.cfg
        H, L = K.shape[0], K.shape[1]
        assert 1 <= L <= self.max_seq_len and int(self.seq_len[b].item()) == 0
        G, R = cfg.group_k, cfg.residual
        npg = (L + 127) // 128
        top = int(self.top[0].item())
        assert npg <= top
        self.page_table[b, :npg] = self.free_pages[top - npg:top].flip(0)
        self.top[0] = top - npg
        nkq, nvq = kivi_segments(L, R)
        d = self.desc()
        for h in range(H):
            if nkq:
                kvq.kv_quant_key_paged(cfg, d, K[h, :nkq].contiguous(), nkq // G, 0, b, h, stream)
            if nvq:
                kvq.kv_quant_value_paged(cfg, d, V[h, :nvq].contiguous(), nvq, 0, b, h, stream)
            _slot_copy(self.k_res[b, h], K[h, nkq:L], [t % R for t in range(nkq, L)])
            _slot_copy(self.v_res[b, h], V[h, nvq:L], [t % R for t in range(nvq, L)])
        self.seq_len[b] = L

    def nbytes_read(self, lens) -> int:
        """Algorithmic bytes of one decode step (as the dense cache: codes, (s, z), fp16 residual)."""
        cfg = self.cfg
        tot = 0
        for L in lens:
            nkq, nvq = kivi_segments(int(L), cfg.residual)
            tot += nkq * D * cfg.bits_k // 8 + (nkq // cfg.group_k) * D * 4
            tot += nvq * D * cfg.bits_v // 8 + nvq * (D // cfg.group_v) * 4
            tot += (int(L) - nkq + int(L) - nvq) * D * 2
        return tot * cfg.n_kv_heads


class KittyCache:
    def __init__(self, cfg: kvq.kvq_config, batch: int, max_seq_len: int, device="cuda"):
        self.cfg, self.batch, self.max_seq_len = cfg, batch, max_seq_len
        H, G, S, R = cfg.n_kv_heads, cfg.group_k, cfg.sink, cfg.residual
        self.kpb = kvq.kvq_kitty_key_page_bytes(cfg)
        self.vpb = kvq.kvq_kitty_value_page_bytes(cfg)
        self.page_cap = max(1, (max(max_seq_len - S, 0) + G - 1) // G)
        self.k_pages = torch.zeros((batch, H, self.page_cap, self.kpb), dtype=torch.uint8, device=device)
        self.v_pages = torch.zeros((batch, H, self.page_cap, self.vpb), dtype=torch.uint8, device=device)
        self.k_sink = torch.zeros((batch, H, max(S, 1), D), dtype=torch.float16, device=device)
        self.v_sink = torch.zeros((batch, H, max(S, 1), D), dtype=torch.float16, device=device)
        self.k_qbuf = torch.zeros((batch, H, G, D), dtype=torch.float16, device=device)
        self.v_qbuf = torch.zeros((batch, H, G, D), dtype=torch.float16, device=device)
        self.v_local = torch.zeros((batch, H, R, D), dtype=torch.float16, device=device)
        self.seq_len = torch.ones(batch, dtype=torch.int32, device=device)

    def fill(self, b: int, kvh: int, K: torch.Tensor, V: torch.Tensor, score_mode: int = 0, stream=None):
        cfg = self.cfg
        L = K.shape[0]
        assert 1 <= L <= self.max_seq_len
        G, S, R = cfg.group_k, cfg.sink, cfg.residual
        pk, nkb, pv, nvb, nloc = kitty_segments(L, G, S, R)
        if pk:
            kvq.kv_quant_key_kitty(cfg, K[S:S + pk * G].contiguous(), pk, score_mode, self.k_pages[b, kvh], stream)
        if pv:
            kvq.kv_quant_value_kitty(cfg, V[S:S + pv * G].contiguous(), pv, self.v_pages[b, kvh], stream)
        ns = min(L, S)
        if ns:
            self.k_sink[b, kvh, :ns] = K[:ns]
            self.v_sink[b, kvh, :ns] = V[:ns]
        k0 = S + pk * G
        if L > k0:
            _slot_copy(self.k_qbuf[b, kvh], K[k0:L], [(t - S) % G for t in range(k0, L)])
        v0 = S + pv * G
        if nvb:
            _slot_copy(self.v_qbuf[b, kvh], V[v0:v0 + nvb], [(t - S) % G for t in range(v0, v0 + nvb)])
        if nloc:
            _slot_copy(self.v_local[b, kvh], V[L - nloc:L], [t % R for t in range(L - nloc, L)])
        self.seq_len[b] = L

    def desc(self) -> kvq.kvq_kitty_cache:
        return kvq.kvq_kitty_cache(self.batch, self.max_seq_len, self.seq_len.data_ptr(), self.k_pages.data_ptr(),
                                   self.v_pages.data_ptr(), self.k_sink.data_ptr(), self.v_sink.data_ptr(),
                                   self.k_qbuf.data_ptr(), self.v_qbuf.data_ptr(), self.v_local.data_ptr())

    def nbytes_read(self, lens) -> int:
        cfg = self.cfg
        tot = 0
        for L in lens:
            pk, nkb, pv, nvb, nloc = kitty_segments(int(L), cfg.group_k, cfg.sink, cfg.residual)
            ns = min(int(L), cfg.sink)
            tot += pk * self.kpb + pv * self.vpb + (2 * ns + nkb + nvb + nloc) * D * 2
        return tot * cfg.n_kv_heads


class KittyPagedCache:
    """Paged Kitty cache of one layer: key and value page records in pools of n_pages pages shared by all
    requests (one page id per 128 tokens after the sink, for every kv head), a page table per request, a
    free-page stack, and per-(row, kv head) fp16 sink, Q-buffers and local window."""

    def __init__(self, cfg: kvq.kvq_config, batch: int, max_seq_len: int, n_pages: int, device="cuda"):
        self.cfg, self.batch, self.max_seq_len, self.n_pages = cfg, batch, max_seq_len, n_pages
        H, G, S, R = cfg.n_kv_heads, cfg.group_k, cfg.sink, cfg.residual
        self.kpb = kvq.kvq_kitty_key_page_bytes(cfg)
        self.vpb = kvq.kvq_kitty_value_page_bytes(cfg)
        self.page_cap = max(1, (max(max_seq_len - S, 0) + G - 1) // G)
        self.k_pages = torch.zeros((n_pages, H, self.kpb), dtype=torch.uint8, device=device)
        self.v_pages = torch.zeros((n_pages, H, self.vpb), dtype=torch.uint8, device=device)
        self.page_table = torch.full((batch, self.page_cap), -1, dtype=torch.int32, device=device)
        self.k_sink = torch.zeros((batch, H, max(S, 1), D), dtype=torch.float16, device=device)
        self.v_sink = torch.zeros((batch, H, max(S, 1), D), dtype=torch.float16, device=device)
        self.k_qbuf = torch.zeros((batch, H, G, D), dtype=torch.float16, device=device)
        self.v_qbuf = torch.zeros((batch, H, G, D), dtype=torch.float16, device=device)
        self.v_local = torch.zeros((batch, H, R, D), dtype=torch.float16, device=device)
        self.seq_len = torch.zeros(batch, dtype=torch.int32, device=device)
        self.free_pages = torch.empty(n_pages, dtype=torch.int32, device=device)
        self.top = torch.zeros(4, dtype=torch.int32, device=device)
        kvq.kv_slot_pool_init(self.pool())

    def pool(self) -> kvq.kvq_slot_pool:
        return kvq.kvq_slot_pool(self.n_pages, self.free_pages.data_ptr(), self.top.data_ptr())

    def desc(self) -> kvq.kvq_kitty_cache:
        return kvq.kvq_kitty_cache(self.batch, self.max_seq_len, self.seq_len.data_ptr(), self.k_pages.data_ptr(),
                                   self.v_pages.data_ptr(), self.k_sink.data_ptr(), self.v_sink.data_ptr(),
                                   self.k_qbuf.data_ptr(), self.v_qbuf.data_ptr(), self.v_local.data_ptr(),
                                   self.page_table.data_ptr(), self.n_pages)

    def shuffle_free(self, perm):
        """Reorder the free stack by a permutation of its entries (host setup)."""
        top = int(self.top[0].item())
        free = self.free_pages[:top].flip(0)
        idx = torch.as_tensor(perm, dtype=torch.int64, device=free.device)
        self.free_pages[:top] = free[idx].flip(0)

    def fill(self, b: int, K: torch.Tensor, V: torch.Tensor, score_mode: int = 0, stream=None):
        """Request b from fp16 K, V [Hkv][L][D]: pops a page for every 128 tokens after the sink that hold
        a token, quantizes the full key / value pages of every head into them."""
        cfg = self.cfg
        H, L = K.shape[0], K.shape[1]
        G, S, R = cfg.group_k, cfg.sink, cfg.residual
        assert 1 <= L <= self.max_seq_len and int(self.seq_len[b].item()) == 0
        npg = (max(L - S, 0) + G - 1) // G
        top = int(self.top[0].item())
        assert npg <= top
        if npg:
            self.page_table[b, :npg] = self.free_pages[top - npg:top].flip(0)
            self.top[0] = top - npg
        pk, nkb, pv, nvb, nloc = kitty_segments(L, G, S, R)
        d = self.desc()
        for h in range(H):
            if pk:
                kvq.kv_quant_key_kitty_paged(cfg, d, K[h, S:S + pk * G].contiguous(), pk, 0, b, h, score_mode,
                                             stream)
            if pv:
                kvq.kv_quant_value_kitty_paged(cfg, d, V[h, S:S + pv * G].contiguous(), pv, 0, b, h, stream)
            ns = min(L, S)
            if ns:
                self.k_sink[b, h, :ns] = K[h, :ns]
                self.v_sink[b, h, :ns] = V[h, :ns]
            k0 = S + pk * G
            if L > k0:
                _slot_copy(self.k_qbuf[b, h], K[h, k0:L], [(t - S) % G for t in range(k0, L)])
            v0 = S + pv * G
            if nvb:
                _slot_copy(self.v_qbuf[b, h], V[h, v0:v0 + nvb], [(t - S) % G for t in range(v0, v0 + nvb)])
            if nloc:
                _slot_copy(self.v_local[b, h], V[h, L - nloc:L], [t % R for t in range(L - nloc, L)])
        self.seq_len[b] = L

    def nbytes_read(self, lens) -> int:
        cfg = self.cfg
        tot = 0
        for L in lens:
            pk, nkb, pv, nvb, nloc = kitty_segments(int(L), cfg.group_k, cfg.sink, cfg.residual)
            ns = min(int(L), cfg.sink)
            tot += pk * self.kpb + pv * self.vpb + (2 * ns + nkb + nvb + nloc) * D * 2
        return tot * cfg.n_kv_heads


class Int8Cache:
    def __init__(self, cfg: kvq.kvq_config, batch: int, max_seq_len: int, layer: int = 0, seed: int = 0,
                 device="cuda"):
        self.cfg, self.batch, self.max_seq_len, self.layer, self.seed = cfg, batch, max_seq_len, layer, seed
        H, T = cfg.n_kv_heads, cfg.int8_block
        self.blk_cap = max(1, (max_seq_len + T - 1) // T)
        self.k_codes = torch.zeros((batch, H, max_seq_len, D), dtype=torch.int8, device=device)
        self.v_codes = torch.zeros((batch, H, max_seq_len, D), dtype=torch.int8, device=device)
        self.k_scale = torch.zeros((batch, H, self.blk_cap, D), dtype=torch.float16, device=device)
        self.v_scale = torch.zeros((batch, H, self.blk_cap, D), dtype=torch.float16, device=device)
        self.k_tail = torch.zeros((batch, H, T, D), dtype=torch.float16, device=device)
        self.v_tail = torch.zeros((batch, H, T, D), dtype=torch.float16, device=device)
        self.seq_len = torch.ones(batch, dtype=torch.int32, device=device)
        self.req_id = torch.zeros(batch, dtype=torch.int32, device=device)

    def fill(self, b: int, kvh: int, K: torch.Tensor, V: torch.Tensor, req_id: int, stream=None):
        cfg = self.cfg
        L = K.shape[0]
        T = cfg.int8_block
        nb, ntail = int8_segments(L, T)
        if nb:
            dev = K.device
            req = torch.full((nb,), req_id, dtype=torch.int32, device=dev)
            head = torch.full((nb,), kvh, dtype=torch.int32, device=dev)
            tok0 = torch.arange(0, nb * T, T, dtype=torch.int32, device=dev)
            for sel, X, codes, scale in ((0, K, self.k_codes, self.k_scale), (1, V, self.v_codes, self.v_scale)):
                kvq.kv_quant_int8_dither(cfg, X[:nb * T].contiguous(), nb, req, head, tok0, self.layer, sel,
                                         self.seed, codes[b, kvh], scale[b, kvh], stream)
        q0 = nb * T
        _slot_copy(self.k_tail[b, kvh], K[q0:L], [t % T for t in range(q0, L)])
        _slot_copy(self.v_tail[b, kvh], V[q0:L], [t % T for t in range(q0, L)])
        self.seq_len[b] = L
        self.req_id[b] = req_id

    def desc(self) -> kvq.kvq_int8_cache:
        return kvq.kvq_int8_cache(self.batch, self.max_seq_len, self.seq_len.data_ptr(), self.req_id.data_ptr(),
                                  self.layer, self.seed, self.k_codes.data_ptr(), self.v_codes.data_ptr(),
                                  self.k_scale.data_ptr(), self.v_scale.data_ptr(), self.k_tail.data_ptr(),
                                  self.v_tail.data_ptr())

    def nbytes_read(self, lens) -> int:
        T = self.cfg.int8_block
        tot = 0
        for L in lens:
            nb, ntail = int8_segments(int(L), T)
            tot += 2 * (nb * T * D + nb * D * 2 + ntail * D * 2)
        return tot * self.cfg.n_kv_heads


class Int8TokenCache:
    """Token-granular INT8 KV pool of one layer: n_slots token slots shared by
    all requests, a per-request slot table and a free-slot stack (the device
    state of kv_append_int8_token / kv_release_int8_token)."""

    def __init__(self, cfg: kvq.kvq_config, batch: int, max_seq_len: int, n_slots: int, layer: int = 0,
                 seed: int = 0, device="cuda"):
        self.cfg, self.batch, self.max_seq_len, self.n_slots = cfg, batch, max_seq_len, n_slots
        self.layer, self.seed = layer, seed
        H, Gc = cfg.n_kv_heads, cfg.int8_group
        self.k_codes = torch.zeros((n_slots, H, D), dtype=torch.int8, device=device)
        self.v_codes = torch.zeros((n_slots, H, D), dtype=torch.int8, device=device)
        self.k_scale = torch.zeros((n_slots, H, D // Gc), dtype=torch.float16, device=device)
        self.v_scale = torch.zeros((n_slots, H, D // Gc), dtype=torch.float16, device=device)
        self.slot_table = torch.full((batch, max_seq_len), -1, dtype=torch.int32, device=device)
        self.seq_len = torch.zeros(batch, dtype=torch.int32, device=device)
        self.free_slots = torch.empty(n_slots, dtype=torch.int32, device=device)
        self.top = torch.zeros(4, dtype=torch.int32, device=device)
        kvq.kv_slot_pool_init(self.pool())

    def pool(self) -> kvq.kvq_slot_pool:
        return kvq.kvq_slot_pool(self.n_slots, self.free_slots.data_ptr(), self.top.data_ptr())

    def desc(self) -> kvq.kvq_int8_token_cache:
        return kvq.kvq_int8_token_cache(self.batch, self.max_seq_len, self.seq_len.data_ptr(),
                                        self.slot_table.data_ptr(), self.n_slots, self.layer, self.seed,
                                        self.k_codes.data_ptr(), self.v_codes.data_ptr(), self.k_scale.data_ptr(),
                                        self.v_scale.data_ptr())

    def shuffle_free(self, perm_pages, page: int = 16):
        """Reorder the free stack by pages of `page` slots (a permutation of the pages, host setup), so that
        later pops hand out scattered pages as a long-running allocator would."""
        top = int(self.top[0].item())
        free = self.free_slots[:top].flip(0)                      # pop order
        n = top // page * page
        idx = torch.as_tensor(perm_pages, dtype=torch.int64, device=free.device)
        pages = free[:n].view(-1, page)[idx].reshape(-1)
        self.free_slots[:top] = torch.cat([pages, free[n:]]).flip(0)

    def fill(self, b: int, K: torch.Tensor, V: torch.Tensor, stream=None):
        """Append L tokens K, V fp16 [L][Hkv][D] to request b (slots popped from the free stack)."""
        L = K.shape[0]
        L0 = int(self.seq_len[b].item())
        top = int(self.top[0].item())
        assert L0 + L <= self.max_seq_len and L <= top
        slots = self.free_slots[top - L:top].flip(0).contiguous()
        self.top[0] = top - L
        kvq.kv_quant_int8_token(self.cfg, self.desc(), K.contiguous(), L, slots, 0, stream)
        kvq.kv_quant_int8_token(self.cfg, self.desc(), V.contiguous(), L, slots, 1, stream)
        self.slot_table[b, L0:L0 + L] = slots
        self.seq_len[b] = L0 + L

    def nbytes_read(self, lens) -> int:
        """Bytes a decode must read: codes and scales of K and V per (token, kv head), plus the slot table."""
        per_tok = self.cfg.n_kv_heads * 2 * (D + 2 * (D // self.cfg.int8_group)) + 4
        return int(sum(int(L) for L in lens)) * per_tok
