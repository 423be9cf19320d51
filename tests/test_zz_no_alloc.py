"""The allocation-free decode entry point (kv_decode_attn_noalloc).

It exists for callers that cannot hand the library a workspace (their own
pool owns all device memory, or no device allocation is allowed after
start-up).  It must give the same outputs as kv_decode_attn with a caller
workspace, call after call, even though every call reuses the same fixed
scratch array inside the library.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

from tests.gpu_util import assert_attn_close, lib, max_abs



@pytest.fixture(scope="module")
def K():
    return lib()


def test_noalloc_rejects_problems_beyond_its_scratch(K):
    """Too large for the fixed scratch: a clear status, nothing launched (host-side check)."""
    cfg = K.make_config(n_q_heads=64, n_kv_heads=8)
    n, need = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, 64, 131072)
    assert need > (16 << 20)
    cache = K.kvq_kivi_cache(64, 131072, 16, 16, 16, 16, 16, 16, 16)
    st = K.raw_call("kv_decode_attn_noalloc", ctypes.byref(cfg), ctypes.byref(cache), 16, 16, None)
    assert st == K.KVQ_ERR_WORKSPACE


def _kivi_cache(K, rng, cfg, B, L, step):
    import torch
    from bit_kv_cache_keyquant_gb300 import cache as C
    cache = C.KiviCache(cfg, B, L, device="cuda")
    for b in range(B):
        for h in range(cfg.n_kv_heads):
            Lb = L - step * b
            cache.fill(b, h, torch.from_numpy(rng.standard_normal((Lb, 128)).astype(np.float16)).cuda(),
                       torch.from_numpy(rng.standard_normal((Lb, 128)).astype(np.float16)).cuda())
    q = torch.from_numpy(rng.standard_normal((B, cfg.n_q_heads, 128)).astype(np.float16)).cuda()
    return cache, q


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice(K):
    """Two calls in a row give the workspace call's output.  Between them a call on another problem
    (more rows, more splits, other lengths) fills the shared scratch with its own partial results, so
    the second call shows that nothing a previous call left in the array is read."""
    import torch
    rng = np.random.default_rng(41)
    cfg = K.make_config(n_q_heads=8, n_kv_heads=4)
    B, L = 3, 1500
    cache, q = _kivi_cache(K, rng, cfg, B, L, 311)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, 8, 128), dtype=torch.float16, device="cuda")
    K.kv_decode_attn(cfg, cache.desc(), q, ref, ws, wsb)
    other_cfg = K.make_config(n_q_heads=4, n_kv_heads=4)
    other, other_q = _kivi_cache(K, rng, other_cfg, 5, 9000, 977)
    n_a, _ = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, L)
    n_b, _ = K.kv_decode_attn_plan(other_cfg, K.KVQ_VARIANT_KIVI, 5, 9000)
    assert n_b > n_a
    outs = []
    for i in range(2):
        out = torch.full((B, 8, 128), float("nan"), dtype=torch.float16, device="cuda")
        K.kv_decode_attn_noalloc(cfg, cache.desc(), q, out)
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy())
        if i == 0:
            junk = torch.empty((5, 4, 128), dtype=torch.float16, device="cuda")
            K.kv_decode_attn_noalloc(other_cfg, other.desc(), other_q, junk)
            torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    r = ref.float().cpu().numpy()
    for o in outs:
        assert np.isfinite(o).all()
        assert_attn_close(o, r)
        assert np.array_equal(o, r)          # the same kernels on the same plan: identical bits
