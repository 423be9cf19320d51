"""Pins of the CPU oracle against things other than itself (CPU only).

Library routines (numpy's IEEE fp16 conversion, numpy textbook attention),
closed forms (lossless quantization of grid-aligned inputs, V == 1, K == 0,
residual-only caches), brute force on tiny inputs, invariants the pages fix
(|x - x^| <= s/2 with the stored fp16 scale; codes in range; no INT8
clipping) and worked numbers printed on the pages (tests/golden).
"""
import json
import os

import numpy as np
import pytest

from bit_kv_cache_keyquant_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")


def f16(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16)


# --------------------------------------------------------------------------
# fp16 conversion
# --------------------------------------------------------------------------
def _special_doubles(rng):
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 70000.0, -65520.0,
            2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25,
            1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1e-10, 3.14159]
    vals += list(rng.standard_normal(3000) * 10.0 ** rng.uniform(-9, 5, 3000))
    # exact ties of fp16 rounding
    h = rng.integers(0, 0x7BFF, 500).astype(np.uint16)
    a = f16(h).astype(np.float64)
    b = f16(h + 1).astype(np.float64)
    vals += list((a + b) / 2)
    return np.array(vals, dtype=np.float64)


def test_half_rn_matches_numpy(orc):
    rng = np.random.default_rng(1)
    for x in _special_doubles(rng):
        want = np.array(x, dtype=np.float64).astype(np.float16).view(np.uint16)
        got = orc.double_to_half(float(x), orc.RN)
        assert got == int(want), (x, hex(got), hex(int(want)))


def test_half_decode_matches_numpy(orc):
    for bits in list(range(0, 0x7C01, 7)) + [0x7BFF, 0x0001, 0x03FF, 0x0400, 0x8001, 0xFBFF]:
        assert orc.half_to_double(bits) == float(f16(bits))


def test_half_directed_rounding_brackets(orc):
    rng = np.random.default_rng(2)
    for x in _special_doubles(rng):
        if abs(x) > 65504:
            continue
        lo = orc.double_to_half(float(x), orc.RD)
        hi = orc.double_to_half(float(x), orc.RU)
        vlo, vhi = orc.half_to_double(lo), orc.half_to_double(hi)
        assert vlo <= x <= vhi
        if vlo == x:
            assert vhi == x
        else:
            # adjacent fp16 values
            assert np.nextafter(np.float16(vlo), np.float16(np.inf)) == np.float16(vhi)


# --------------------------------------------------------------------------
# affine quantizer
# --------------------------------------------------------------------------
@pytest.mark.parametrize("bits", [2, 4])
def test_affine_error_bound_and_range(orc, bits):
    rng = np.random.default_rng(3 + bits)
    qmax = (1 << bits) - 1
    for trial in range(300):
        n = int(rng.integers(2, 40))
        scale = 10.0 ** rng.uniform(-4, 3)
        x = (rng.standard_normal(n) * scale + rng.uniform(-3, 3) * scale).astype(np.float16)
        if trial % 7 == 0:
            x[:] = x[0]                      # constant group
        s, z = orc.affine_fit(x, bits)
        sv, zv = orc.half_to_double(s), orc.half_to_double(z)
        xv = x.astype(np.float64)
        assert zv <= xv.min()
        assert zv + qmax * sv >= xv.max()
        for xb, xx in zip(x.view(np.uint16), xv):
            code = orc.affine_code(int(xb), s, z, bits)
            assert 0 <= code <= qmax
            xhat = code * sv + zv
            assert abs(xx - xhat) <= sv / 2 * (1 + 2 ** -20) + (0 if sv else 0.0)
        if xv.max() > xv.min():
            # s is the fp16 round-up of the fp32 step, raised only as far as coverage needs
            s32 = np.float32(np.float32(xv.max()) - np.float32(zv)) / np.float32(qmax)
            assert sv >= float(s32)
            prev = orc.half_to_double(s - 1)
            assert prev < float(s32) or zv + qmax * prev < xv.max()


def test_affine_grid_aligned_is_lossless(orc):
    rng = np.random.default_rng(5)
    for _ in range(200):
        bits = int(rng.choice([2, 4]))
        qmax = (1 << bits) - 1
        s = 2.0 ** int(rng.integers(-6, 3))
        z = s * int(rng.integers(-40, 40))
        n = int(rng.integers(4, 33))
        k = rng.integers(0, qmax + 1, n)
        k[0], k[1] = 0, qmax
        x = (z + k * s).astype(np.float16)
        assert np.all(x.astype(np.float64) == z + k * s)
        sb, zb = orc.affine_fit(x, bits)
        assert orc.half_to_double(sb) == s and orc.half_to_double(zb) == z
        for xb, kk in zip(x.view(np.uint16), k):
            assert orc.affine_code(int(xb), sb, zb, bits) == kk


def test_affine_brute_force_requantize(orc):
    """All 4^4 code tuples of a 4-token 2-bit group: dequantize, refit, same codes."""
    s = 0.25
    z = -1.5
    for idx in range(256):
        k = [(idx >> (2 * i)) & 3 for i in range(4)]
        x = np.array([z + kk * s for kk in k], dtype=np.float16)
        sb, zb = orc.affine_fit(x, 2)
        if min(k) == max(k):
            assert orc.half_to_double(sb) == 0.0
            continue
        sv, zv = orc.half_to_double(sb), orc.half_to_double(zb)
        codes = [orc.affine_code(int(b), sb, zb, 2) for b in x.view(np.uint16)]
        xhat = [c * sv + zv for c in codes]
        assert np.allclose(xhat, x.astype(np.float64), atol=sv / 2 + 1e-12)
        if min(k) == 0 and max(k) == 3:
            assert codes == k


def test_kitty_step_examples(orc):
    g = json.load(open(GOLDEN))["kitty_step_examples"]
    for lo, hi, step, tol in g["cases"]:
        x = np.linspace(lo, hi, 16).astype(np.float16)
        s, z = orc.affine_fit(x, 2)
        assert abs(orc.half_to_double(s) - step) <= tol
        assert orc.half_to_double(z) == lo


# --------------------------------------------------------------------------
# packing layouts
# --------------------------------------------------------------------------
def test_kivi_key_layout_is_a_lane_friendly_bijection(orc):
    seen = {}
    for t in range(64):
        for c in range(128):
            off = orc.kivi_key_byte_offset(t, c)
            seen.setdefault((off, orc.kivi_key_bit(t)), set()).add((t, c))
            # a byte holds tokens q, q+8, q+16, q+24 of one channel (q = t % 8);
            # the 32 bytes of (q, r) are chunk 4q+r of each 512-byte half and
            # cover channels 16k + 2r + {0, 1, 8, 9}, k = 0..7, in word k % 4
            q, r, k = t % 8, (c % 8) // 2, c // 16
            assert (off % 512) // 16 == 4 * q + r
            assert (off % 1024) // 512 == k // 4 and (off % 16) // 4 == k % 4
            assert off // 1024 == t // 32
            assert orc.kivi_key_bit(t) == 2 * ((t % 32) // 8)
    assert sorted({o for o, _ in seen}) == list(range(2048))
    assert all(len(v) == 1 for v in seen.values())
    # (s, z) storage order: chunk row r's 32 channels are the 8-entry chunks r, 4+r, 8+r, 12+r,
    # word k of the codes at entries (k%2)*4 + byte of chunk (k/2)*4 + r
    idx = [orc.kivi_key_sz_index(c) for c in range(128)]
    assert sorted(idx) == list(range(128))
    for c in range(128):
        k, r = c // 16, (c % 8) // 2
        byte = (orc.kivi_key_byte_offset(0, c) % 16) % 4
        assert idx[c] == ((k // 2) * 4 + r) * 8 + (k % 2) * 4 + byte


def test_kivi_key_layout_4bit_is_a_lane_friendly_bijection(orc):
    """4-bit keys: a 32-token tile is two 1024-byte planes; plane p // 2 holds the tokens q + 8p of the
    2-bit byte at bits 4 (p % 2), so a lane still finds its tokens x channels in the same chunks."""
    seen = {}
    for t in range(64):
        for c in range(128):
            off, bit = orc.kivi_key_byte_offset(t, c, 4), orc.kivi_key_bit(t, 4)
            seen.setdefault((off, bit), set()).add((t, c))
            p = (t % 32) // 8
            assert off // 2048 == t // 32 and (off % 2048) // 1024 == p // 2
            assert off % 1024 == orc.kivi_key_byte_offset(t % 8, c) and bit == 4 * (p % 2)
    assert sorted({o for o, _ in seen}) == list(range(4096))
    assert all(len(v) == 1 for v in seen.values()) and len(seen) == 64 * 128


def test_kivi_value_layout_is_a_lane_friendly_bijection(orc):
    """2-bit KIVI values in 32-token tiles in the fragment order of a tensor-core value product: a byte
    holds four channels 32g + 4q + {0..3} of one token; word 4q + r of a 16-token half holds that byte
    (g, q) of tokens r, r + 4, r + 8, r + 12; lane 4q + r's 16 bytes are its words for g = 0..3."""
    seen = set()
    for t in range(64):
        for c in range(128):
            off, bit = orc.kivi_value_byte_offset(t, c), orc.kivi_value_bit(c)
            tt, g, q = t % 32, c // 32, (c % 32) // 4
            assert off // 1024 == t // 32 and (off % 1024) // 512 == tt // 16
            assert (off % 512) // 16 == 4 * q + tt % 4            # the lane's 16 bytes
            assert (off % 16) // 4 == g and off % 4 == (tt % 16) // 4
            assert bit == 2 * (c % 4)
            seen.add((off, bit))
    assert len(seen) == 64 * 128 and {o for o, _ in seen} == set(range(2048))


def test_kivi_value_layout_4bit_pairs_channels_of_one_token(orc):
    """4-bit KIVI value tiles: a byte holds channels c and c + 64 of one token (so tokens are written
    independently); word 2m + w of lane 4q + r's 32 bytes of a 16-token half holds channels 16m + q
    (bytes 0, 1) and 16m + q + 8 (bytes 2, 3) of tokens r + 8w, r + 8w + 4 in its low nibbles, the same
    channels + 64 in its high nibbles."""
    seen = set()
    for t in range(64):
        for c in range(128):
            off, bit = orc.kivi_value_byte_offset4(t, c), orc.kivi_value_bit4(c)
            tt, c64 = t % 32, c % 64
            assert off // 2048 == t // 32 and (off % 2048) // 1024 == tt // 16
            assert (off % 1024) // 32 == 4 * (c64 % 8) + tt % 4                # the lane's 32 bytes
            assert (off % 32) // 4 == 2 * (c64 // 16) + (tt // 8) % 2          # word 2m + w
            assert off % 4 == 2 * ((c64 // 8) % 2) + (tt // 4) % 2 and bit == 4 * (c // 64)
            seen.add((off, bit))
    assert len(seen) == 64 * 128 and {o for o, _ in seen} == set(range(4096))
    by_byte = {}
    for t in range(32):
        for c in range(128):
            by_byte.setdefault(orc.kivi_value_byte_offset4(t, c), set()).add(t)
    assert all(len(v) == 1 for v in by_byte.values())                     # one token per byte


def test_kivi_value_pack_roundtrip_and_tail(orc):
    rng = np.random.default_rng(66)
    for n in (1, 31, 32, 45, 96):
        codes = rng.integers(0, 4, (n, 128)).astype(np.uint8)
        packed = orc.kivi_value_pack(codes, 2, tiles=True)
        assert packed.shape == ((n + 31) // 32 * 32, 32)
        flat = packed.reshape(-1)
        got = np.zeros_like(codes)
        written = np.zeros(flat.size, bool)
        for t in range(n):
            for c in range(128):
                o = orc.kivi_value_byte_offset(t, c)
                got[t, c] = (flat[o] >> orc.kivi_value_bit(c)) & 3
                written[o] = True
        assert np.array_equal(got, codes)
        assert not flat[~written].any()                        # tokens past n leave zero bytes
        # without tiles: one token-major row per token, as tokenmajor_pack
        assert np.array_equal(orc.kivi_value_pack(codes, 2), orc.tokenmajor_pack(codes, 2))
        c4 = rng.integers(0, 16, (n, 128)).astype(np.uint8)
        assert np.array_equal(orc.kivi_value_pack(c4, 4), orc.tokenmajor_pack(c4, 4))
        # 4-bit tiles
        p4 = orc.kivi_value_pack(c4, 4, tiles=True)
        assert p4.shape == ((n + 31) // 32 * 32, 64)
        f4 = p4.reshape(-1)
        got4 = np.zeros_like(c4)
        written4 = np.zeros(f4.size, bool)
        for t in range(n):
            for c in range(128):
                o = orc.kivi_value_byte_offset4(t, c)
                got4[t, c] = (f4[o] >> orc.kivi_value_bit4(c)) & 15
                written4[o] = True
        assert np.array_equal(got4, c4) and not f4[~written4].any()


def test_kivi_decode_reads_both_value_layouts(orc):
    """The same cache stored with value tiles or token-major decodes to the same binary64 output."""
    rng = np.random.default_rng(67)
    L = 333
    K = rng.standard_normal((L, 128)).astype(np.float16)
    V = (rng.standard_normal((L, 128)) * 10 ** rng.uniform(-1, 1, 128)).astype(np.float16)
    q = rng.standard_normal((2, 128)).astype(np.float16)
    a = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V), L=L)
    b = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V, value_tiles=True), L=L, value_tiles=True)
    assert np.array_equal(a, b)
    a4 = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V, bits_v=4), L=L, bits_v=4)
    b4 = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V, bits_v=4, value_tiles=True), L=L, bits_v=4,
                             value_tiles=True)
    assert np.array_equal(a4, b4)
    # and the tile bytes are read as tiles: a decode told the wrong layout differs
    c = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V, value_tiles=True), L=L)
    assert not np.allclose(a, c, atol=1e-3)


@pytest.mark.parametrize("bits", [2, 4])
def test_kivi_key_pack_roundtrip_any_width(orc, bits):
    rng = np.random.default_rng(60 + bits)
    codes = rng.integers(0, 1 << bits, (3, 64, 128)).astype(np.uint8)
    packed = orc.kivi_key_pack(codes, bits)
    assert packed.shape == (3, 64 * 128 * bits // 8)
    for g in range(3):
        for t in range(0, 64, 5):
            for c in range(0, 128, 3):
                byte = int(packed[g, orc.kivi_key_byte_offset(t, c, bits)])
                assert (byte >> orc.kivi_key_bit(t, bits)) & ((1 << bits) - 1) == codes[g, t, c]


def test_tokenmajor_pack_4bit_matches_numpy_nibbles(orc):
    rng = np.random.default_rng(64)
    codes = rng.integers(0, 16, (9, 128)).astype(np.uint8)
    packed = orc.tokenmajor_pack(codes, 4)
    assert np.array_equal(packed, (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))


@pytest.mark.parametrize("bk,bv", [(4, 4), (4, 2), (2, 4)])
def test_grid_aligned_cache_equals_fp_attention_any_width(orc, bk, bv):
    """Inputs on the b-bit grid are lossless at both widths, which pins the 4-bit unpacking of
    keys and values in the decode."""
    rng = np.random.default_rng(70 + 10 * bk + bv)
    L = 300
    kmax, vmax = (1 << bk) - 1, (1 << bv) - 1
    kk = rng.integers(0, kmax + 1, (L, 128))
    kk[::32][:, :] = 0
    kk[1::32][:, :] = kmax                  # every 32-token group spans codes 0..kmax
    ks = 2.0 ** rng.integers(-4, -1, 128)
    K = (ks * (kk - 2)).astype(np.float16)
    vk = rng.integers(0, vmax + 1, (L, 128))
    vk[:, ::32] = 0
    vk[:, 1::32] = vmax
    V = (0.0625 * vk - 0.25).astype(np.float16)
    q = rng.standard_normal((2, 128)).astype(np.float16)
    parts = orc.kivi_build_one(K, V, bits_k=bk, bits_v=bv)
    assert parts[0].shape[1] == 32 * 128 * bk // 8 and parts[2].shape[1] == 128 * bv // 8
    out = orc.kivi_decode_one(q, *parts, L=L, bits_k=bk, bits_v=bv)
    for h in range(2):
        assert np.allclose(out[h], textbook(q[h], K, V, 128 ** -0.5), atol=1e-12, rtol=0)
    # and the 2-bit reading of the same 4-bit bytes is not the same cache
    if bk == 4:
        wrong = orc.kivi_decode_one(q, *parts, L=L, bits_k=2, bits_v=bv) if parts[0].size else None
        assert wrong is None or not np.allclose(wrong, out, atol=1e-6)


def test_kivi_key_pack_roundtrip(orc):
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 4, (3, 64, 128)).astype(np.uint8)
    packed = orc.kivi_key_pack(codes)
    for g in range(3):
        for t in range(64):
            for c in range(0, 128, 5):
                b = packed[g, orc.kivi_key_byte_offset(t, c)]
                assert (b >> orc.kivi_key_bit(t)) & 3 == codes[g, t, c]
    sz = rng.integers(0, 65536, (3, 128, 2)).astype(np.uint16)
    st = orc.kivi_key_sz_pack(sz)
    for c in range(128):
        assert np.array_equal(st[:, orc.kivi_key_sz_index(c)], sz[:, c, 0])
        assert np.array_equal(st[:, 128 + orc.kivi_key_sz_index(c)], sz[:, c, 1])


def test_tokenmajor_pack_matches_numpy_bitops(orc):
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 4, (50, 128)).astype(np.uint8)
    packed = orc.tokenmajor_pack(codes)
    c4 = codes.reshape(50, 32, 4).astype(np.uint32)
    want = (c4[..., 0] | (c4[..., 1] << 2) | (c4[..., 2] << 4) | (c4[..., 3] << 6)).astype(np.uint8)
    assert np.array_equal(packed, want)


# --------------------------------------------------------------------------
# Kitty
# --------------------------------------------------------------------------
def _page(rng, G=128, D=128, heavy=True):
    sig = 10.0 ** rng.uniform(-1, 1, D) if heavy else np.ones(D)
    return (rng.standard_normal((G, D)) * sig).astype(np.float16)


def test_kitty_topk_brute_force(orc):
    rng = np.random.default_rng(8)
    for trial in range(6):
        x = _page(rng)
        if trial == 1:
            x[:, 5] = x[:, 9]                           # exact tie: lower index wins
        score = np.abs(x.astype(np.float64)).sum(axis=0)  # exact: < 2^53 units of 2^-24
        order = sorted(range(128), key=lambda c: (-score[c], c))
        want = np.zeros(128, np.uint8)
        want[order[:16]] = 1
        assert np.array_equal(orc.kitty_select(x, 16, 0), want)
        # variance mode, sequential fp32 sums in token order
        s1 = np.zeros(128, np.float32)
        s2 = np.zeros(128, np.float32)
        for t in range(128):
            v = x[t].astype(np.float32)
            s1 = s1 + v
            s2 = s2 + v * v
        m = s1 / np.float32(128)
        var = s2 / np.float32(128) - m * m
        order = sorted(range(128), key=lambda c: (-float(var[c]), c))
        want = np.zeros(128, np.uint8)
        want[order[:16]] = 1
        assert np.array_equal(orc.kitty_select(x, 16, 1), want)


def test_kitty_planes_combine_to_4bit_codes(orc):
    rng = np.random.default_rng(9)
    x = _page(rng)
    page = orc.kitty_key_page(x, 16)
    assert page.size == 5248
    codes, s, z = orc.kitty_key_page_decode(page, 128, 128, 16)
    boosted = orc.kitty_select(x, 16, 0)
    idx = page[4096 + 512:4096 + 512 + 128]
    assert np.array_equal(np.flatnonzero(idx < 16), np.flatnonzero(boosted))
    assert sorted(idx[idx < 16].tolist()) == list(range(16))
    assert np.all(idx[boosted == 0] == 17)
    for c in range(128):
        bits = 4 if boosted[c] else 2
        sc, zc = orc.affine_fit(x[:, c], bits)
        assert (s[c], z[c]) == (sc, zc)
        for t in range(0, 128, 3):
            assert codes[t, c] == orc.affine_code(int(x[t, c].view(np.uint16)), sc, zc, bits)


def test_kitty_plane_order_is_lane_friendly(orc):
    """Key-page planes in the fragment order of the KIVI 2-bit key tiles (the Kitty page fixes the
    planes, not the byte order inside them): the low plane of a 128-token page is four 1024-byte
    tiles where a byte holds tokens q, q+8, q+16, q+24 of one channel and lane 4q + r's 16-byte
    chunks hold channels 16k + 2r + {0, 1, 8, 9}; the high plane gives each 32-token tile a block of
    Kp * 8 bytes (Kp = K rounded up to 4) whose 4-byte word 8r + q of 16-row block kh holds rows
    16kh + 4r + {0..3} at tokens q + 8p."""
    seen = set()
    for t in range(128):
        for c in range(128):
            off, bit = orc.kitty_low_byte_offset(t, c), orc.kitty_code_bit(t)
            q, p, r, k = t % 8, (t % 32) // 8, (c % 8) // 2, c // 16
            e, h = c % 2, (c % 16) // 8
            assert off // 1024 == t // 32 and bit == 2 * p
            assert (off % 1024) // 512 == k // 4 and (off % 512) // 16 == 4 * q + r
            assert (off % 16) // 4 == k % 4 and off % 4 == e + 2 * h
            seen.add((off, bit))
    assert len(seen) == 128 * 128 and {o for o, _ in seen} == set(range(4096))
    for K in (1, 3, 4, 13, 16, 17, 32, 92):
        Kp = orc.kitty_high_rows(K)
        assert Kp % 4 == 0 and K <= Kp < K + 4
        seen = set()
        for t in range(128):
            for rho in range(Kp):
                off = orc.kitty_high_byte_offset(K, t, rho)
                j, q = t // 32, t % 8
                assert j * Kp * 8 <= off < (j + 1) * Kp * 8           # the tile's block
                o = off - j * Kp * 8
                assert o // 128 == rho // 16 and (o % 128) // 32 == (rho % 16) // 4
                assert (o % 32) // 4 == q and o % 4 == rho % 4
                seen.add((off, orc.kitty_code_bit(t)))
        assert len(seen) == 128 * Kp and {o for o, _ in seen} == set(range(Kp * 32))


def test_kitty_page_planes_are_kivi_tiles_of_the_codes(orc):
    """The low plane equals the KIVI 2-bit key packing of the page's low code bits; the high plane
    holds the high bits of the boosted channels by rank, zero in rows K..Kp-1."""
    rng = np.random.default_rng(12)
    x = _page(rng)
    for K in (13, 16):
        page = orc.kitty_key_page(x, K)
        Kp = orc.kitty_high_rows(K)
        assert page.size == 4096 + Kp * 32 + 128 + 512
        codes, _, _ = orc.kitty_key_page_decode(page, 128, 128, K)
        low = orc.kivi_key_pack((codes & 3).reshape(1, 128, 128), 2).reshape(-1)
        assert np.array_equal(page[:4096], low)
        boosted = np.flatnonzero(orc.kitty_select(x, K, 0))
        high = page[4096:4096 + Kp * 32]
        for rho in range(Kp):
            for t in range(128):
                v = (int(high[orc.kitty_high_byte_offset(K, t, rho)]) >> orc.kitty_code_bit(t)) & 3
                assert v == (codes[t, boosted[rho]] >> 2 if rho < K else 0)


def test_kitty_alpha_limits(orc):
    rng = np.random.default_rng(10)
    x = _page(rng)
    # alpha = 0: plain per-channel 2-bit over G = 128 tokens
    page0 = orc.kitty_key_page(x, 0)
    c0, s0, z0 = orc.kitty_key_page_decode(page0, 128, 128, 0)
    kc, ksz = orc.kivi_key_codes(x[None], 2)
    assert np.array_equal(c0, kc[0]) and np.array_equal(s0, ksz[0, :, 0]) and np.array_equal(z0, ksz[0, :, 1])
    # alpha = 1: uniform 4-bit
    page1 = orc.kitty_key_page(x, 128)
    c1, s1, z1 = orc.kitty_key_page_decode(page1, 128, 128, 128)
    kc4, ksz4 = orc.kivi_key_codes(x[None], 4)
    assert np.array_equal(c1, kc4[0]) and np.array_equal(s1, ksz4[0, :, 0])


def test_page_byte_accounts(orc):
    g = json.load(open(GOLDEN))
    D = G = 128
    for key in ("kitty_bits_per_element", "kitty_pro_bits_per_element"):
        a = g[key]["alpha"]
        K = int(round(a * D))
        code_bits = (D * G * 2 + K * G * 2) / (D * G)
        assert code_bits == g[key]["value"]
    assert g["kitty_boosted_channels"]["K"] == [int(a * 128) for a in g["kitty_boosted_channels"]["alpha"]]
    assert orc.kitty_key_page_bytes(128, 128, 16) == 4096 + 512 + 128 + 512
    assert orc.kitty_key_page_bytes(128, 128, 13) == orc.kitty_key_page_bytes(128, 128, 16)
    assert orc.kitty_value_page_bytes(128, 128) == 4096 + 512
    # INT8 block cache: 128 one-byte codes plus 128 fp16 scales per 256 tokens
    assert 128 + 128 * 2 / 256 == g["int8_block_bytes_per_token_per_side"]["value"]
    # token-granular variant: 128 codes plus one fp16 scale per 32 channels
    assert 128 + (128 // 32) * 2 == g["int8_token_granular_bytes_per_token_per_side"]["value"]
    assert g["kivi_group_defaults"]["R"] % g["kivi_group_defaults"]["G"] == 0


# --------------------------------------------------------------------------
# Philox / dither
# --------------------------------------------------------------------------
def test_philox_inverse_roundtrip(orc):
    rng = np.random.default_rng(11)
    ctrs = [[0, 0, 0, 0], [0xFFFFFFFF] * 4, [0x80000000, 1, 0xFFFFFFFF, 7]]
    ctrs += rng.integers(0, 2 ** 32, (200, 4), dtype=np.uint64).tolist()
    for ctr in ctrs:
        key = rng.integers(0, 2 ** 32, 2, dtype=np.uint64)
        out = orc.philox(ctr, key)
        back = orc.philox_inverse(out, key)
        assert [int(v) for v in back] == [int(v) for v in ctr]


def test_dither_statistics_and_uniqueness(orc):
    vals = np.array([orc.dither(0x1234, 5, 3, kv, 2, t, c)
                     for kv in (0, 1) for t in range(64) for c in range(128)], dtype=np.float64)
    n = vals.size
    assert np.all(vals >= -0.5) and np.all(vals < 0.5)
    assert abs(vals.mean()) < 5 * np.sqrt(1 / 12 / n)
    assert abs(vals.var() - 1 / 12) < 0.004
    # distinct five-tuples give distinct draws (collisions of 24-bit values are rare)
    assert len(set(vals.tolist())) > 0.99 * n
    # the K and V streams differ; changing request, layer or head changes the stream
    a = orc.dither(7, 1, 2, 0, 3, 100, 17)
    assert a != orc.dither(7, 1, 2, 1, 3, 100, 17)
    assert a != orc.dither(7, 2, 2, 0, 3, 100, 17)
    assert a != orc.dither(7, 1, 3, 0, 3, 100, 17)
    assert a != orc.dither(7, 1, 2, 0, 4, 100, 17)
    assert a != orc.dither(8, 1, 2, 0, 3, 100, 17)


def test_int8_dither_no_clip_and_error_bound(orc):
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((256, 128)) * 10.0 ** rng.uniform(-2, 2, 128)).astype(np.float16)
    x[:, 3] = 0                                    # all-zero channel: s = 0
    codes, scale = orc.int8_quant_block(x, 99, 4, 1, 0, 2, 512)
    assert scale[3] == 0 and np.all(codes[:, 3] == 0)
    assert np.all(np.abs(codes.astype(np.int32)) <= 127)
    for c in range(0, 128, 9):
        s = orc.half_to_double(int(scale[c]))
        amax = np.abs(x[:, c].astype(np.float64)).max()
        assert s == float(np.float16(np.float32(amax) / np.float32(126.5)))
        for t in range(0, 256, 17):
            xi = orc.dither(99, 4, 1, 0, 2, 512 + t, c)
            xhat = orc.half_to_double(0) if s == 0 else s * (int(codes[t, c]) - xi)
            assert abs(float(x[t, c]) - xhat) <= s / 2 * (1 + 2 ** -20) + 1e-30


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def textbook(q, K, V, sm):
    s = (K.astype(np.float64) @ q.astype(np.float64)) * sm
    p = np.exp(s - s.max())
    p /= p.sum()
    return p @ V.astype(np.float64)


def test_residual_only_is_textbook_attention(orc):
    rng = np.random.default_rng(13)
    for L in (1, 5, 77, 128):
        K = rng.standard_normal((L, 128)).astype(np.float16)
        V = rng.standard_normal((L, 128)).astype(np.float16)
        q = rng.standard_normal((2, 128)).astype(np.float16)
        parts = orc.kivi_build_one(K, V)
        out = orc.kivi_decode_one(q, *parts, L=L)
        for h in range(2):
            assert np.allclose(out[h], textbook(q[h], K, V, 128 ** -0.5), atol=1e-12, rtol=0)


def test_grid_aligned_cache_equals_fp_attention(orc):
    """Inputs on the quantization grid: every quantized segment is lossless."""
    rng = np.random.default_rng(14)
    L = 300
    kk = rng.integers(0, 4, (L, 128))
    kk[::32][:, :] = 0
    kk[1::32][:, :] = 3                     # every 32-token group spans codes 0..3
    ks = 2.0 ** rng.integers(-3, 1, 128)
    K = (ks * (kk - 1)).astype(np.float16)
    vk = rng.integers(0, 4, (L, 128))
    vk[:, ::32] = 0
    vk[:, 1::32] = 3                        # every 32-channel group spans 0..3
    V = (0.125 * vk - 0.25).astype(np.float16)
    q = rng.standard_normal((1, 128)).astype(np.float16)
    out = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V), L=L)
    assert np.allclose(out[0], textbook(q[0], K, V, 128 ** -0.5), atol=1e-12, rtol=0)


def test_constant_values_and_zero_keys(orc):
    rng = np.random.default_rng(15)
    L = 400
    K = rng.standard_normal((L, 128)).astype(np.float16)
    V = np.ones((L, 128), np.float16)
    q = rng.standard_normal((3, 128)).astype(np.float16)
    out = orc.kivi_decode_one(q, *orc.kivi_build_one(K, V), L=L)
    assert np.allclose(out, 1.0, atol=1e-12)
    # K == 0: uniform softmax, output = mean of the dequantized values
    K0 = np.zeros((L, 128), np.float16)
    V2 = rng.standard_normal((L, 128)).astype(np.float16)
    parts = orc.kivi_build_one(K0, V2)
    out = orc.kivi_decode_one(q, *parts, L=L)
    nkq, nvq = orc.kivi_segments(L)
    codes, sz = orc.kivi_value_codes(V2[:nvq])
    s = sz[..., 0].view(np.float16).astype(np.float64)
    z = sz[..., 1].view(np.float16).astype(np.float64)
    vhat = codes.reshape(nvq, 4, 32) * s[..., None] + z[..., None]
    allv = np.concatenate([vhat.reshape(nvq, 128), V2[nvq:].astype(np.float64)])
    assert np.allclose(out, allv.mean(axis=0)[None], atol=1e-12)


def test_kitty_and_int8_short_contexts_are_textbook(orc):
    rng = np.random.default_rng(16)
    for L in (1, 31, 32, 33, 160):
        K = rng.standard_normal((L, 128)).astype(np.float16)
        V = rng.standard_normal((L, 128)).astype(np.float16)
        q = rng.standard_normal((4, 128)).astype(np.float16)
        out = orc.kitty_decode_one(q, *orc.kitty_build_one(K, V), L=L)
        for h in range(4):
            assert np.allclose(out[h], textbook(q[h], K, V, 128 ** -0.5), atol=1e-12)
    for L in (1, 100, 256):
        K = rng.standard_normal((L, 128)).astype(np.float16)
        V = rng.standard_normal((L, 128)).astype(np.float16)
        q = rng.standard_normal((2, 128)).astype(np.float16)
        parts = orc.int8_build_one(K, V, 5, 9, 0, 1)
        out = orc.int8_decode_one(q, *parts, L=L, seed=5, request=9, layer=0, kv_head=1)
        for h in range(2):
            assert np.allclose(out[h], textbook(q[h], K, V, 128 ** -0.5), atol=1e-12)


def test_kitty_segments_match_mixed_key_workload(orc):
    # 131072 tokens: 1023 key pages + 96 buffered keys; 1022 value pages +
    # 96 buffered + 128 local values; 32 sink tokens each side
    assert orc.kitty_segments(131072) == (1023, 96, 1022, 96, 128)
    assert orc.kivi_segments(4096) == (3968, 3968)


def test_int8_request_id_not_batch_position(orc):
    """Permuting batch rows together with their request ids leaves outputs unchanged."""
    rng = np.random.default_rng(17)
    L = 600
    rows = [(rng.standard_normal((L, 128)).astype(np.float16),
             rng.standard_normal((L, 128)).astype(np.float16),
             rng.standard_normal((2, 128)).astype(np.float16), rid) for rid in (11, 42)]
    outs = {}
    for order in ((0, 1), (1, 0)):
        for pos, i in enumerate(order):
            K, V, q, rid = rows[i]
            parts = orc.int8_build_one(K, V, 3, rid, 2, 0)
            outs[(order, rid)] = orc.int8_decode_one(q, *parts, L=L, seed=3, request=rid, layer=2, kv_head=0)
    for rid in (11, 42):
        assert np.array_equal(outs[((0, 1), rid)], outs[((1, 0), rid)])


def test_int8_quantized_attention_error_is_small(orc):
    """Dithered INT8 with the no-clip scale stays close to fp attention."""
    rng = np.random.default_rng(18)
    L = 700
    K = rng.standard_normal((L, 128)).astype(np.float16)
    V = rng.standard_normal((L, 128)).astype(np.float16)
    q = rng.standard_normal((2, 128)).astype(np.float16)
    parts = orc.int8_build_one(K, V, 1, 2, 3, 4)
    out = orc.int8_decode_one(q, *parts, L=L, seed=1, request=2, layer=3, kv_head=4)
    for h in range(2):
        assert np.max(np.abs(out[h] - textbook(q[h], K, V, 128 ** -0.5))) < 5e-3


def _int8_block_xhat(orc, codes, scale, X, nq, seed, request, layer, kv_sel, kv_head, T=256):
    """Dequantized tokens of one side of a block-INT8 cache, element by element: s (code - xi) with the
    writer's five-tuple dither (request, layer, kv_sel, kv head, absolute token, channel) for the quantized
    tokens, the fp16 token itself for the active block."""
    out = X.astype(np.float64).copy()
    for t in range(nq):
        for c in range(128):
            s = orc.half_to_double(int(scale[t // T, c]))
            out[t, c] = s * (int(codes[t, c]) - orc.dither(seed, request, layer, kv_sel, kv_head, t, c))
    return out


def test_int8_decode_equals_attention_over_block_dequantized_tokens(orc):
    """WitCert sec. 6.1 read side: the block-INT8 decode equals textbook attention over keys and values
    dequantized element by element as s (code - xi), xi regenerated from the writer's tuple, over two
    quantized 256-token blocks and an fp16 active block (L = 700: 512 quantized + 188 fp16)."""
    rng = np.random.default_rng(51)
    L, seed, request, layer, kv_head = 700, 0x0123456789AB, 77, 3, 5
    K = (rng.standard_normal((L, 128)) * 3).astype(np.float16)
    V = (rng.standard_normal((L, 128)) * 2).astype(np.float16)
    q = rng.standard_normal((3, 128)).astype(np.float16)
    kc, vc, ks, vs, kt, vt = orc.int8_build_one(K, V, seed, request, layer, kv_head)
    nq = 512                                       # ((L - 1) mod 256) + 1 = 188 tokens stay fp16
    out = orc.int8_decode_one(q, kc, vc, ks, vs, kt, vt, L=L, seed=seed, request=request, layer=layer,
                              kv_head=kv_head)
    khat = _int8_block_xhat(orc, kc, ks, K, nq, seed, request, layer, 0, kv_head)
    vhat = _int8_block_xhat(orc, vc, vs, V, nq, seed, request, layer, 1, kv_head)
    # the fp16 active block is read as is; the quantized tokens are not (the dither moves them)
    assert np.array_equal(khat[nq:], K[nq:].astype(np.float64))
    assert np.max(np.abs(khat[:nq] - K[:nq].astype(np.float64))) > 1e-3
    for h in range(3):
        assert np.allclose(out[h], textbook(q[h], khat, vhat, 128 ** -0.5), rtol=0, atol=1e-12)
    # the pin has the power to see a wrong read-side stream: the K / V streams swapped, or the token index
    # taken relative to its block, each move the textbook result far beyond 1e-12
    k_swap = _int8_block_xhat(orc, kc, ks, K, nq, seed, request, layer, 1, kv_head)
    v_swap = _int8_block_xhat(orc, vc, vs, V, nq, seed, request, layer, 0, kv_head)
    assert np.max(np.abs(textbook(q[0], k_swap, v_swap, 128 ** -0.5) - out[0])) > 1e-6
    v_rel = vhat.copy()
    for t in range(256, nq):
        for c in range(128):
            s = orc.half_to_double(int(vs[1, c]))
            v_rel[t, c] = s * (int(vc[t, c]) - orc.dither(seed, request, layer, 1, kv_head, t - 256, c))
    assert np.max(np.abs(textbook(q[0], khat, v_rel, 128 ** -0.5) - out[0])) > 1e-6


def _fp32_decode(Kh, V, q, sm):
    """Attention with every product exact and rounded once to fp32, the logits summed over channels in
    fp32 in channel order, and the softmax in fp32: the best any fp32-accumulating decode can do."""
    q32 = (q * sm).astype(np.float32)
    K32 = Kh.astype(np.float32)
    s = np.zeros(Kh.shape[0], np.float32)
    for c in range(Kh.shape[1]):
        s = (s + K32[:, c] * q32[c]).astype(np.float32)
    p = np.exp((s - s.max()).astype(np.float32)).astype(np.float32)
    return (p / p.sum()) @ V.astype(np.float32)


def test_fp32_accumulation_limit_on_extreme_query_ranges(orc):
    """Reading of the tolerance: max-abs 2e-3 with fp32 accumulation holds while the logits stay moderate.
    A query of 6e4 in one channel over channels of 1e-2 makes logits of about 2e4 whose ties (2-bit codes
    tie many tokens on the large channel) are broken by differences of about 1e-2: even exact products
    summed in fp32 miss 2e-3 there, while at 3e3 over 1e-3 (logits of about 800) they stay within half of it."""
    rng = np.random.default_rng(22)
    L, sm = 1280, 128 ** -0.5
    worst = {}
    for big, small in ((6e4, 1e-2), (3e3, 1e-3)):
        errs = []
        for _ in range(3):
            K = rng.standard_normal((L, 128)).astype(np.float16)
            V = rng.standard_normal((L, 128)).astype(np.float16)
            codes, sz = orc.kivi_key_codes(K.reshape(L // 32, 32, 128))
            s_ = f16(sz[..., 0].copy()).astype(np.float64)
            z_ = f16(sz[..., 1].copy()).astype(np.float64)
            Kh = (codes.astype(np.float64) * s_[:, None, :] + z_[:, None, :]).reshape(L, 128)
            q = rng.standard_normal(128) * small
            q[5] = big
            q = q.astype(np.float16).astype(np.float64)
            errs.append(np.max(np.abs(_fp32_decode(Kh, V, q, sm) - textbook(q, Kh, V, sm))))
        worst[big] = max(errs)
    assert worst[6e4] > 2e-3
    assert worst[3e3] < 1e-3


# --------------------------------------------------------------------------
# token-granular INT8 over a slot pool (WitCert, SGLang storage subsection)
# --------------------------------------------------------------------------
def _int8t_xhat(orc, codes, scale, Gc, seed, layer, kv_sel, kv_head, slot):
    return np.array([orc.half_to_double(int(scale[c // Gc])) *
                     (int(codes[c]) - orc.dither_slot(seed, layer, kv_sel, kv_head, slot, c))
                     for c in range(len(codes))])


@pytest.mark.parametrize("Gc", [32, 64, 128])
def test_int8t_scale_per_token_group_bound_and_no_clip(orc, Gc):
    rng = np.random.default_rng(40 + Gc)
    for trial in range(6):
        x = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 3, 128)).astype(np.float16)
        if trial == 0:
            x[:Gc] = 0                                  # an all-zero group: s = 0, codes 0
        slot = int(rng.integers(0, 2 ** 31 - 1))
        codes, scale = orc.int8t_quant_token(x, Gc, 77, 5, trial & 1, 3, slot)
        assert scale.shape == (128 // Gc,)
        for g in range(128 // Gc):
            amax = np.abs(x[g * Gc:(g + 1) * Gc].astype(np.float64)).max()
            assert scale[g] == np.float16(np.float32(amax) / np.float32(126.5)).view(np.uint16)
        # no clipping: |x/s + xi| < 127.07 always rounds inside [-127, 127]; the extreme codes stay reachable
        assert np.all(np.abs(codes.astype(np.int32)) <= 127)
        xhat = _int8t_xhat(orc, codes, scale, Gc, 77, 5, trial & 1, 3, slot)
        s = np.array([orc.half_to_double(int(scale[c // Gc])) for c in range(128)])
        assert np.all(np.abs(x.astype(np.float64) - xhat) <= s / 2 * (1 + 2 ** -20) + 1e-30)
        if trial == 0:
            assert np.all(codes[:Gc] == 0) and scale[0] == 0 and np.all(xhat[:Gc] == 0)


def test_int8t_groups_are_independent(orc):
    """Changing one group's channels leaves every other group's scale and codes unchanged."""
    rng = np.random.default_rng(47)
    x = rng.standard_normal(128).astype(np.float16)
    a_codes, a_scale = orc.int8t_quant_token(x, 32, 1, 0, 0, 0, 1234)
    y = x.copy()
    y[64:96] *= np.float16(40)
    b_codes, b_scale = orc.int8t_quant_token(y, 32, 1, 0, 0, 0, 1234)
    keep = np.r_[0:64, 96:128]
    assert np.array_equal(a_codes[keep], b_codes[keep])
    assert a_scale[0] == b_scale[0] and a_scale[1] == b_scale[1] and a_scale[3] == b_scale[3]
    assert a_scale[2] != b_scale[2]


def test_int8t_dither_is_keyed_by_slot_unbiased_and_uniform(orc):
    """Subtractive dither: over many slots the error x^ - x of a fixed value is uniform on
    [-s/2, s/2) (mean 0, variance s^2/12) whatever x is; the stream depends on the slot only."""
    x = np.zeros(128, np.float16)
    x[0] = np.float16(126.5 * 0.01)                     # fixes s of group 0 near 0.01
    x[1:32] = np.linspace(-1.2, 1.2, 31).astype(np.float16)
    errs = []
    for slot in range(1500):
        codes, scale = orc.int8t_quant_token(x, 32, 9, 1, 0, 2, slot)
        s = orc.half_to_double(int(scale[0]))
        xhat = _int8t_xhat(orc, codes[:32], scale, 32, 9, 1, 0, 2, slot)
        errs.append((xhat - x[:32].astype(np.float64)) / s)
    e = np.array(errs)
    assert np.all(np.abs(e) <= 0.5 * (1 + 2 ** -20))
    n = e.shape[0]
    assert np.all(np.abs(e.mean(axis=0)) < 4 * np.sqrt(1 / 12 / n))
    assert np.all(np.abs(e.var(axis=0) - 1 / 12) < 0.012)
    # the counter carries the slot, not the position: the same slot gives the same codes
    c1, _ = orc.int8t_quant_token(x, 32, 9, 1, 0, 2, 700)
    c2, _ = orc.int8t_quant_token(x, 32, 9, 1, 0, 2, 700)
    c3, _ = orc.int8t_quant_token(x, 32, 9, 1, 0, 2, 701)
    assert np.array_equal(c1, c2) and not np.array_equal(c1, c3)
    # distinct (layer, kv_sel, kv_head, slot) give distinct streams
    seen = {tuple(orc.dither_slot(9, la, ks, h, sl, c) for c in range(4))
            for la in range(3) for ks in range(2) for h in range(3) for sl in (0, 1, 2 ** 31 - 1)}
    assert len(seen) == 3 * 2 * 3 * 3


def _int8t_pool(n_slots, Hkv, Gc=32):
    return (np.zeros((n_slots, Hkv, 128), np.int8), np.zeros((n_slots, Hkv, 128), np.int8),
            np.zeros((n_slots, Hkv, 128 // Gc), np.uint16), np.zeros((n_slots, Hkv, 128 // Gc), np.uint16))


def test_int8t_decode_gathers_by_slot(orc):
    """One token: attention returns its dequantized value (within s/2 of v); K == 0 gives the mean of
    the dequantized values of the request's own slots, even with other slots holding large values."""
    rng = np.random.default_rng(48)
    Hkv, n_slots = 2, 300
    pool = _int8t_pool(n_slots, Hkv)
    junk = (rng.standard_normal((n_slots, 128)) * 1000).astype(np.float16)
    for h in range(Hkv):
        orc.int8t_write(pool, junk, junk, range(n_slots), h, 32, 5, 7)
    # one token at slot 123 of kv head 1
    k1 = rng.standard_normal((1, 128)).astype(np.float16)
    v1 = rng.standard_normal((1, 128)).astype(np.float16)
    orc.int8t_write(pool, k1, v1, [123], 1, 32, 5, 7)
    q = rng.standard_normal((2, 128)).astype(np.float16)
    o = orc.int8t_decode_one(q, pool, [123], 1, 5, 7)
    s = np.repeat([orc.half_to_double(int(z)) for z in pool[3][123, 1]], 32)
    for h in range(2):
        assert np.all(np.abs(o[h] - v1[0].astype(np.float64)) <= s / 2 * (1 + 2 ** -20))
    # K == 0 over a scattered request
    L = 40
    slots = rng.permutation(n_slots)[:L]
    V = rng.standard_normal((L, 128)).astype(np.float16)
    orc.int8t_write(pool, np.zeros((L, 128), np.float16), V, slots, 0, 32, 5, 7)
    o = orc.int8t_decode_one(q, pool, slots, 0, 5, 7)
    vhat = np.array([_int8t_xhat(orc, pool[1][s_, 0], pool[3][s_, 0], 32, 5, 7, 1, 0, int(s_)) for s_ in slots])
    for h in range(2):
        assert np.allclose(o[h], vhat.mean(axis=0), rtol=0, atol=1e-12)
        assert np.max(np.abs(o[h] - V.astype(np.float64).mean(axis=0))) < 0.02


def test_int8t_decode_equals_attention_over_slot_dequantized_tokens(orc):
    """The decode equals textbook attention over keys and values dequantized element by element from
    the request's slots with the dither of each slot (s (code - xi), evaluated here in numpy)."""
    rng = np.random.default_rng(50)
    Hkv, n_slots, L = 3, 400, 60
    pool = _int8t_pool(n_slots, Hkv)
    slots = rng.permutation(n_slots)[:L]
    K = (rng.standard_normal((L, 128)) * 4).astype(np.float16)
    V = rng.standard_normal((L, 128)).astype(np.float16)
    orc.int8t_write(pool, K, V, slots, 2, 32, 21, 4)
    q = rng.standard_normal((2, 128)).astype(np.float16)
    o = orc.int8t_decode_one(q, pool, slots, 2, 21, 4)
    khat = np.array([_int8t_xhat(orc, pool[0][s_, 2], pool[2][s_, 2], 32, 21, 4, 0, 2, int(s_)) for s_ in slots])
    vhat = np.array([_int8t_xhat(orc, pool[1][s_, 2], pool[3][s_, 2], 32, 21, 4, 1, 2, int(s_)) for s_ in slots])
    for h in range(2):
        sc = khat @ q[h].astype(np.float64) * 128 ** -0.5
        p = np.exp(sc - sc.max())
        assert np.allclose(o[h], (p / p.sum()) @ vhat, rtol=0, atol=1e-12)


def test_int8t_attention_close_to_fp(orc):
    rng = np.random.default_rng(49)
    L, n_slots = 500, 2048
    pool = _int8t_pool(n_slots, 1)
    K = rng.standard_normal((L, 128)).astype(np.float16)
    V = rng.standard_normal((L, 128)).astype(np.float16)
    slots = rng.permutation(n_slots)[:L]
    orc.int8t_write(pool, K, V, slots, 0, 32, 11, 2)
    q = rng.standard_normal((3, 128)).astype(np.float16)
    out = orc.int8t_decode_one(q, pool, slots, 0, 11, 2)
    for h in range(3):
        assert np.max(np.abs(out[h] - textbook(q[h], K, V, 128 ** -0.5))) < 5e-3


# --------------------------------------------------------------------------
# synthetic input generator
# --------------------------------------------------------------------------
def test_inputs_distribution_and_determinism():
    w = I.WORKLOADS[3]
    a = I.gen_kv_np(w, I.T_V, 5, 3, 4096)
    b = I.gen_kv_np(w, I.T_V, 5, 3, 1000, row0=3096)
    assert np.array_equal(a[3096:], b)
    x = a.astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.02
    k = I.gen_kv_np(w, I.T_K, 5, 3, 512).astype(np.float64)
    gain = I.key_channel_gain(w)[3]
    assert np.count_nonzero(gain == 15.0) == 1
    assert k[:, gain == 15.0].std() > 10
    lens = I.seq_lens(I.WORKLOADS[5])
    assert lens.min() >= 16384 and lens.max() <= 65536 and len(set(lens.tolist())) > 1


def test_kitty_grid_aligned_long_context_equals_fp_attention(orc):
    """Keys on {z + 5s*k} are lossless under both the 2-bit (step 5s) and the
    4-bit (step s) fit; values on a per-token 2-bit grid are lossless.  Every
    page, Q-buffer, local-window and sink slot must then carry its own token."""
    rng = np.random.default_rng(19)
    for L in (700, 32 + 128 * 2 + 128 + 1, 32 + 128 * 2 + 128):
        s_c = 2.0 ** rng.integers(-5, -2, 128)
        k = rng.integers(0, 4, (L, 128))
        for p0 in range(32, L, 128):
            k[p0, :] = 0
            if p0 + 1 < L:
                k[p0 + 1, :] = 3
        K = (5 * s_c * k - 0.5).astype(np.float16)
        vk = rng.integers(0, 4, (L, 128))
        vk[:, 0], vk[:, 1] = 0, 3
        st = 2.0 ** rng.integers(-4, -1, L)
        V = (st[:, None] * vk + 0.25).astype(np.float16)
        q = rng.standard_normal((4, 128)).astype(np.float16)
        out = orc.kitty_decode_one(q, *orc.kitty_build_one(K, V), L=L)
        for h in range(4):
            assert np.allclose(out[h], textbook(q[h], K, V, 128 ** -0.5), atol=1e-12, rtol=0)
