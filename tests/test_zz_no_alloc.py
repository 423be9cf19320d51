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


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice(K):
    import torch
    from bit_kv_cache_keyquant_gb300 import cache as C
    rng = np.random.default_rng(41)
    cfg = K.make_config(n_q_heads=8, n_kv_heads=4)
    B, L = 3, 1500
    cache = C.KiviCache(cfg, B, L, device="cuda")
    for b in range(B):
        for h in range(4):
            Lb = L - 311 * b
            cache.fill(b, h, torch.from_numpy(rng.standard_normal((Lb, 128)).astype(np.float16)).cuda(),
                       torch.from_numpy(rng.standard_normal((Lb, 128)).astype(np.float16)).cuda())
    q = torch.from_numpy(rng.standard_normal((B, 8, 128)).astype(np.float16)).cuda()
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, L)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, 8, 128), dtype=torch.float16, device="cuda")
    K.kv_decode_attn(cfg, cache.desc(), q, ref, ws, wsb)
    outs = []
    for _ in range(2):
        out = torch.full((B, 8, 128), float("nan"), dtype=torch.float16, device="cuda")
        K.kv_decode_attn_noalloc(cfg, cache.desc(), q, out)
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy())
    assert K.kvq_get_device_error() == 0
    r = ref.float().cpu().numpy()
    for o in outs:
        assert np.isfinite(o).all()
        assert_attn_close(o, r)
