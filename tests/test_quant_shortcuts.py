"""CPU checks of the arithmetic shortcuts the kernels take, in numpy float32 (IEEE binary32, round to
nearest) and integers against float64 references; no GPU and no oracle code involved.

1. The fit's fix-up test: for fp16 mn <= mx, z = fp16_RD(mn) and an fp16 step s, the exact test
   z + qmax*s < mx equals the fp32 test fl(qmax*s) < fl_up(mx - z) (qmax*s is an fp32 number; no fp32
   number lies strictly between mx - z and its round-up).
2. The element code: rint(fl(d * fl(1/s))) equals rint(fl(d / s)) whenever the product is farther than
   0.5 - 1e-5 from a half-integer (|d / s| <= 32), so only near-ties need the quotient.
3. The per-head decode kernel's dp4a key products (below).
4. The INT8 decode kernel's warp sum through shared memory (below).
"""
import numpy as np


def _f32_round_up(x64):
    """Least float32 >= x64 (x64 a float64 holding an exact value)."""
    f = x64.astype(np.float32)
    lo = f.astype(np.float64) < x64
    f[lo] = np.nextafter(f[lo], np.float32(np.inf))
    return f


def _fp16_rd(x):
    h = x.astype(np.float16)
    hi = h.astype(np.float64) > x
    h[hi] = np.nextafter(h[hi], np.float16(-np.inf))
    return h


def test_fixup_test_exact_in_fp32():
    np.seterr(over="ignore", invalid="ignore")
    rng = np.random.default_rng(1)
    n = 400000
    scale = 10.0 ** rng.uniform(-6, 4.5, n)
    a = (rng.standard_normal(n) * scale).astype(np.float16)
    b = (a.astype(np.float64) + np.abs(rng.standard_normal(n)) * scale * 10.0 ** rng.uniform(-4, 0, n)).astype(np.float16)
    ok = np.isfinite(a) & np.isfinite(b) & (b > a)
    mn, mx = a[ok].astype(np.float64), b[ok].astype(np.float64)
    z = _fp16_rd(mn).astype(np.float64)
    for qmax in (3, 15):
        # candidate steps around the fitted one, as the loop meets them
        s0 = ((mx - z) / qmax).astype(np.float16)
        for k in (-2, -1, 0, 1, 2):
            s = s0.copy()
            for _ in range(abs(k)):
                s = np.nextafter(s, np.float16(np.inf if k > 0 else -np.inf))
            s64 = s.astype(np.float64)
            good = np.isfinite(s64) & (s64 > 0)
            exact = z[good] + qmax * s64[good] < mx[good]
            p32 = (np.float32(qmax) * s[good].astype(np.float32))
            assert np.all(p32.astype(np.float64) == qmax * s64[good])            # p is an fp32 number
            up = _f32_round_up(mx[good] - z[good])
            assert np.array_equal(exact, p32 < up)


def test_fixup_test_at_the_boundary():
    """mx - z one fp16 subnormal above qmax*s: only the rounded-up difference keeps the test exact."""
    np.seterr(over="ignore", invalid="ignore")
    rng = np.random.default_rng(3)
    s = (10.0 ** rng.uniform(-2, 3, 20000)).astype(np.float16)
    for qmax in (3, 15):
        p64 = qmax * s.astype(np.float64)
        mx = p64.astype(np.float16)
        keep = np.isfinite(mx) & (mx.astype(np.float64) == p64)          # qmax*s itself an fp16 number
        for zt in (-2.0 ** -24, -2.0 ** -20, -2.0 ** -14):
            z = np.full(keep.sum(), zt)
            mxk, sk = mx[keep].astype(np.float64), s[keep]
            exact = z + qmax * sk.astype(np.float64) < mxk                  # true: z < 0
            p32 = np.float32(qmax) * sk.astype(np.float32)
            assert exact.all()
            assert np.array_equal(exact, p32 < _f32_round_up(mxk - z))


def test_product_form_code_matches_quotient_off_ties():
    rng = np.random.default_rng(2)
    n = 2000000
    s = (10.0 ** rng.uniform(-7, 4, n) * rng.uniform(0.5, 1.0, n)).astype(np.float16).astype(np.float32)
    s = s[(s > 0) & np.isfinite(s)]
    q = rng.uniform(0.0, 15.5, s.size)
    # quotients spread over [0, 15.5], with a share placed near half-integers
    near = rng.random(s.size) < 0.3
    q[near] = np.floor(q[near]) + 0.5 + rng.uniform(-3e-5, 3e-5, near.sum())
    d = (q * s.astype(np.float64)).astype(np.float32)
    exact = np.rint((d / s).astype(np.float32))
    rinv = (np.float32(1.0) / s).astype(np.float32)
    qa = (d * rinv).astype(np.float32)
    r = np.rint(qa)
    tie = np.abs((qa - r).astype(np.float32)) > np.float32(0.49999)
    assert tie.any() and (~tie).any()
    assert np.array_equal(r[~tie], exact[~tie])


def _key_fixed_exp(wm):
    """The per-head kernel's fixed-point exponent: wm 2^fx in [2^21, 2^22), clamped to [-100, 100]."""
    ex = (np.asarray(wm, dtype=np.float32).view(np.uint32) >> 23) & 255
    return np.clip(148 - ex.astype(np.int64), -100, 100)


def test_dp4a_key_products_reconstruct_the_fixed_point_dot():
    """3. The per-head kernel's key scores: weights alpha q s in 22-bit fixed point against the group's
    largest |weight|, split into two unsigned bytes and a signed top byte; dp4a sums of four
    (u8 code byte) x (weight byte) products, combined as (A0 + 256 A1) + 65536 A2, equal the integer
    dot product exactly, and the result is within 128 * 3 * 2^-22 * max|W| (the weights' rounding) of
    the binary64 dot product."""
    rng = np.random.default_rng(4)
    for trial in range(300):
        w = (rng.standard_normal(128) * 10.0 ** rng.uniform(-3, 3, 128)).astype(np.float32)
        if trial % 7 == 0:
            w[:] = 0.0                                     # an all-zero query: every weight 0
        fx = int(_key_fixed_exp(np.max(np.abs(w))))
        wi = np.rint(w.astype(np.float64) * 2.0 ** fx).astype(np.int64)      # fl(w 2^fx) is exact here
        assert np.all(np.abs(wi) <= 2 ** 22)
        b0, b1 = wi & 0xFF, (wi >> 8) & 0xFF
        b2 = ((wi >> 16) & 0xFF).astype(np.int8).astype(np.int64)            # signed top byte
        assert np.array_equal(b0 + 256 * b1 + 65536 * b2, wi)
        for bits in (2, 4):
            codes = rng.integers(0, 2 ** bits, size=128)
            for slot in range(8 // bits):                  # the code's position in its byte
                x = codes << (bits * slot)                 # the masked byte, an unsigned value
                a0, a1, a2 = (int(np.sum(x * b)) for b in (b0, b1, b2))   # four-byte sums, accumulated
                assert (a0 + (a1 << 8)) < 2 ** 31 and abs(a2) < 2 ** 24
                combined = float(np.float32(a2)) * 65536.0 + float(np.float32(a0 + (a1 << 8)))
                assert a0 + 256 * a1 + 65536 * a2 == int(np.sum(x * wi))
                got = combined * 2.0 ** (-fx - bits * slot)
                want = float(np.sum(codes.astype(np.float64) * w.astype(np.float64)))
                bound = 128 * (2 ** bits - 1) * 0.5 * 2.0 ** -fx + 2 ** -22 * abs(want) + 1e-300
                assert abs(got - want) <= bound


def test_int8_swizzled_column_sum():
    """The INT8 decode kernel sums 32 partials per lane over the warp by storing lane l's 32 floats as
    row l of a 32 x 32 float block, its 16-byte chunk k at chunk position k ^ (l & 7), and letting lane
    L read column L: element (4 * (L >> 2) + (L & 3)) of every row, found at chunk (L >> 2) ^ (l & 7).
    Checked here: the read gives lane L the sum over lanes of partial L (what the register
    reduce-scatter gave), every row is written whole and once, each 16-byte store of a chunk index k
    by the warp touches every one of the 32 banks exactly four times (four wavefronts, the minimum for
    512 bytes), and each column load touches 32 distinct banks (one wavefront)."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal((32, 32)).astype(np.float32)        # v[lane, k]: lane's partial k
    smem = np.full((32, 32), np.nan, dtype=np.float32)
    written = np.zeros((32, 32), dtype=int)
    for k in range(8):                                          # store instruction k, all lanes
        banks = np.zeros(32, dtype=int)
        for lane in range(32):
            pos = 4 * (k ^ (lane & 7))
            smem[lane, pos:pos + 4] = v[lane, 4 * k:4 * k + 4]
            written[lane, pos:pos + 4] += 1
            for w in range(4):
                banks[(lane * 32 + pos + w) % 32] += 1
        assert (banks == 4).all()
    assert (written == 1).all()
    got = np.zeros(32, dtype=np.float64)
    for row in range(32):                                       # load instruction row, all lanes
        addr = [row * 32 + 4 * ((L >> 2) ^ (row & 7)) + (L & 3) for L in range(32)]
        assert len({a % 32 for a in addr}) == 32
        for L in range(32):
            got[L] += smem.reshape(-1)[addr[L]]
    np.testing.assert_allclose(got, v.astype(np.float64).sum(axis=0), rtol=1e-5, atol=1e-5)
