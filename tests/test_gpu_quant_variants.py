"""GPU bit-exactness of the Kitty page quantizers and the INT8 dither writer."""
import numpy as np
import pytest
import torch

from tests.gpu_util import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def K():
    return lib()


def _pages(rng, n, heavy=True):
    sig = 10.0 ** rng.uniform(-1, 1, (n, 1, 128)) if heavy else np.ones((n, 1, 128))
    x = (rng.standard_normal((n, 128, 128)) * sig).astype(np.float16)
    x[0, :, 5] = x[0, :, 9]          # exact score tie between channels 5 and 9
    x[1, :, 3] = np.float16(0.5)     # constant channel
    return x


@pytest.mark.parametrize("Kb", [0, 13, 16, 32, 128])
@pytest.mark.parametrize("mode", [0, 1])
def test_kitty_key_pages_bitexact(K, orc, Kb, mode):
    rng = np.random.default_rng(300 + Kb + mode)
    n = 9
    x = _pages(rng, n)
    cfg = K.make_config(group_k=128, n_q_heads=32, n_kv_heads=8, boost_k=Kb)
    pb = K.kvq_kitty_key_page_bytes(cfg)
    pages = torch.full((n, pb), 0xCD, dtype=torch.uint8, device=DEV)
    K.kv_quant_key_kitty(cfg, torch.from_numpy(x).to(DEV), n, mode, pages)
    torch.cuda.synchronize()
    got = pages.cpu().numpy()
    for p in range(n):
        assert np.array_equal(got[p], orc.kitty_key_page(x[p], Kb, mode)), p


def test_kitty_value_pages_bitexact(K, orc):
    rng = np.random.default_rng(310)
    n = 7
    x = _pages(rng, n, heavy=False)
    cfg = K.make_config(group_k=128, n_q_heads=32, n_kv_heads=8, boost_k=16)
    pb = K.kvq_kitty_value_page_bytes(cfg)
    pages = torch.full((n, pb), 0xCD, dtype=torch.uint8, device=DEV)
    K.kv_quant_value_kitty(cfg, torch.from_numpy(x).to(DEV), n, pages)
    torch.cuda.synchronize()
    got = pages.cpu().numpy()
    for p in range(n):
        assert np.array_equal(got[p], orc.kitty_value_page(x[p])), p


def test_int8_dither_bitexact(K, orc):
    rng = np.random.default_rng(320)
    n, T = 5, 256
    x = (rng.standard_normal((n, T, 128)) * 10.0 ** rng.uniform(-3, 3, (n, 1, 128))).astype(np.float16)
    x[2, :, 17] = 0                                    # all-zero channel: s = 0
    req = np.array([7, 7, 123456789, -5, 0x7FFFFFFF], np.int32)
    head = np.array([0, 3, 1, 7, 2], np.int32)
    tok0 = np.array([0, 256, 1024, 65280, 2 ** 30], np.int32)
    cfg = K.make_config(n_q_heads=64, n_kv_heads=8)
    seed = 0xFEEDFACE12345678
    for sel, layer in ((0, 0), (1, 31), (0, 32767)):
        codes = torch.full((n, T, 128), 99, dtype=torch.int8, device=DEV)
        scale = torch.full((n, 128), -1, dtype=torch.int16, device=DEV)
        K.kv_quant_int8_dither(cfg, torch.from_numpy(x).to(DEV), n, torch.from_numpy(req).to(DEV),
                               torch.from_numpy(head).to(DEV), torch.from_numpy(tok0).to(DEV), layer, sel, seed,
                               codes, scale)
        torch.cuda.synchronize()
        gc = codes.cpu().numpy()
        gs = scale.cpu().numpy().view(np.uint16)
        for b in range(n):
            rc, rs = orc.int8_quant_block(x[b], seed, int(req[b]), layer, sel, int(head[b]), int(tok0[b]))
            assert np.array_equal(gs[b], rs), (sel, b)
            assert np.array_equal(gc[b], rc), (sel, b)
