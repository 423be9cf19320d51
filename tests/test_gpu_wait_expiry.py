"""The KIVI decode kernels' bounded mbarrier waits, made to run out (through the C ABI).

A separate test copy of the library (built with KVQ_FAULT_INJECT; the product
library has no such hook) lets CTA 0's producer leave one stage unfilled and
shortens the waits to 256 tries.  The consumers' waits on that stage must give
up and return: the call completes, the context stays usable, the device error
flag reports KVQ_DEVICE_ERR_WAIT_TIMEOUT, and the next call without the
injection gives the first call's result bit for bit.  Nothing traps and
nothing reads or writes outside its buffers: the unfilled stage is only never
announced, and the producer still waits (bounded) for every copy it issued.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.gpu_util import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    return lib()


@pytest.fixture(scope="module")
def T(tmp_path_factory):
    from bit_kv_cache_keyquant_gb300 import build
    t = ctypes.CDLL(build.build_test_lib(str(tmp_path_factory.mktemp("kvq_test_lib"))))
    t.kvq_test_inject_wait.argtypes = [ctypes.c_int, ctypes.c_uint]
    t.kvq_test_inject_wait.restype = None
    t.kv_decode_attn.restype = ctypes.c_int
    t.kvq_get_device_error.restype = ctypes.c_int
    return t


def _decode(T, cfg, cache, q, wsb):
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device=DEV)
    out = torch.full((cache.batch, cfg.n_q_heads, 128), float("nan"), dtype=torch.float16, device=DEV)
    desc = cache.desc()
    st = T.kv_decode_attn(ctypes.byref(cfg), ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()),
                          ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(wsb),
                          None)
    assert st == 0
    torch.cuda.synchronize()                       # the call completes: no trap, no hang
    flags = ctypes.c_uint32(0)
    assert T.kvq_get_device_error(ctypes.byref(flags)) == 0
    return out.cpu(), flags.value


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2)])       # one head per unit; four heads per unit
def test_bounded_wait_runs_out_and_the_next_call_is_clean(K, T, Hq, Hkv):
    from bit_kv_cache_keyquant_gb300 import cache as C
    rng = np.random.default_rng(61 + Hq)
    B, L = 2, 2000
    cfg = K.make_config(n_q_heads=Hq, n_kv_heads=Hkv)
    cache = C.KiviCache(cfg, B, L, device=DEV)
    for b in range(B):
        for h in range(Hkv):
            cache.fill(b, h, torch.from_numpy(rng.standard_normal((L, 128)).astype(np.float16)).to(DEV),
                       torch.from_numpy(rng.standard_normal((L, 128)).astype(np.float16)).to(DEV))
    q = torch.from_numpy(rng.standard_normal((B, Hq, 128)).astype(np.float16)).to(DEV)
    _, wsb = K.kv_decode_attn_plan(cfg, K.KVQ_VARIANT_KIVI, B, L)

    ref, f0 = _decode(T, cfg, cache, q, wsb)
    assert f0 == 0 and torch.isfinite(ref.float()).all()
    try:
        T.kvq_test_inject_wait(0, 256)             # CTA 0's first stage is never filled
        _, f1 = _decode(T, cfg, cache, q, wsb)
    finally:
        T.kvq_test_inject_wait(-1, 0)
    assert f1 & K.KVQ_DEVICE_ERR_WAIT_TIMEOUT
    again, f2 = _decode(T, cfg, cache, q, wsb)
    assert f2 == 0
    assert torch.equal(again, ref)
    # the product library runs the same kernels: the same bits
    out = torch.empty_like(ref, device=DEV)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    K.kv_decode_attn(cfg, cache.desc(), q, out, ws, wsb)
    torch.cuda.synchronize()
    assert K.kvq_get_device_error() == 0
    assert torch.equal(out.cpu(), ref)
