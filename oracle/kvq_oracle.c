/*
 * kvq_oracle.c -- plain, slow CPU oracle of the quantized-KV decode path.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or call this code.  It
 * shares no source, header, table or helper with the CUDA library; it is
 * written from the method's definitions:
 *
 *   KIVI (zenmind.me "KIVI：key 按通道 / value 按 token ..."), section 3.3:
 *     keys quantized per channel over groups of G tokens, values per token,
 *     a full-precision residual of at most R tokens, attention over the
 *     concatenation of the quantized part and the residual (Eq. 3).
 *   Kitty (paper-graph-ui "Kitty: Accurate and Efficient 2-bit KV Cache
 *     Quantization with Dynamic Channel-wise Precision Boost"): Eq. 2 channel
 *     score, top-K precision boost, the two-plane page decomposition, the
 *     boost index, Algorithm 1 dequantization, sink / Q-buffer / local window.
 *   WitCert (arxiv 2607.28699, section 6): INT8 subtractive dither
 *     x^ = s(round(x/s + xi) - xi), Philox4x32-10 keyed by (request, layer,
 *     KV head, token, channel), block scale s = amax/126.5 stored in fp16 and
 *     used for quantization, split-free softmax.  Its token-granular form
 *     for a slot-paged pool (the SGLang storage subsection): one scale per
 *     token and group of Gc channels, Philox keyed by (layer, KV head, slot,
 *     channel), every token quantized when it is written.
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *     Easy as 1, 2, 3", SC'11 (the published round function and constants).
 *
 * Every float operation is IEEE binary32 or binary64 round-to-nearest-even;
 * the file must be compiled with -ffp-contract=off and without fast-math.
 * Attention is evaluated in binary64 with no splitting.
 *
 * Parity status of each function (see the tests that pin it):
 *   half conversion     pinned (numpy float16 RN, adjacency of RD/RU)
 *   affine quantizer    pinned (error bound, range, grid-aligned lossless, brute force)
 *   packing / unpacking pinned (round trip, brute force against per-element reads)
 *   Kitty selection     pinned (brute-force top-K, alpha=0 / alpha=1 limits)
 *   Philox4x32-10       pinned on the GPU machine against cuRAND's Philox4x32-10;
 *                       on the CPU by its inverse and by uniformity statistics
 *   attention           pinned (R >= L equals textbook softmax attention,
 *                       V == 1, K == 0, permutation invariance)
 *   token-granular INT8 pinned (error bound, no clipping, group locality,
 *                       unbiased and uniform dither error over slots,
 *                       one-token attention, K == 0, slot gather)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* IEEE binary16                                                        */
/* ------------------------------------------------------------------ */

ORC_API double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

enum { ORC_RN = 0, ORC_RD = 1, ORC_RU = 2 };

/* Round a binary64 value to binary16 with the given IEEE rounding
 * direction (nearest-even, toward -inf, toward +inf). */
ORC_API uint16_t orc_double_to_half(double x, int mode)
{
    if (isnan(x))
        return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    /* rounding of the magnitude: 0 = truncate, 1 = away from zero, 2 = nearest-even */
    int how;
    if (mode == ORC_RN)
        how = 2;
    else if (mode == ORC_RD)
        how = sign ? 1 : 0;
    else
        how = sign ? 0 : 1;
    if (isinf(a))
        return sign | 0x7C00;
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);                 /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                /* floor(log2 a) */
    if (E < -14)
        E = -14;                   /* subnormals share the quantum 2^-24 */
    double quantum = ldexp(1.0, E - 10);
    double qv = a / quantum;       /* exact: division by a power of two */
    double fl = floor(qv);
    double frac = qv - fl;
    double r;
    if (frac == 0.0 || how == 0)
        r = fl;
    else if (how == 1)
        r = fl + 1.0;
    else if (frac > 0.5)
        r = fl + 1.0;
    else if (frac < 0.5)
        r = fl;
    else
        r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * quantum;
    if (v > 65504.0)
        return (how == 0) ? (uint16_t)(sign | 0x7BFF) : (uint16_t)(sign | 0x7C00);
    if (v < ldexp(1.0, -14))
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    frexp(v, &e2);
    E = e2 - 1;
    int mant = (int)(v / ldexp(1.0, E - 10)) - 1024;
    return sign | (uint16_t)(((E + 15) << 10) | mant);
}

static uint16_t half_next_up_positive(uint16_t h) { return (uint16_t)(h + 1); }

/* ------------------------------------------------------------------ */
/* Asymmetric min-max affine quantizer (Kitty Observation 1 formula,    */
/* Kitty "Quantization Step"; KIVI section 3.1 zero point / scale)      */
/* ------------------------------------------------------------------ */

/* Fit (s, z) to n fp16 values x[i*stride] for b-bit codes.
 *   z = fp16 rounded toward -inf of min
 *   s = fp16 rounded toward +inf of fp32 (max - z) / (2^b - 1),
 *       then raised by one fp16 step while z + s*(2^b-1) < max (exact test)
 *   max == min gives s = 0 (every code 0, dequantized value z = x). */
ORC_API void orc_affine_fit(const uint16_t *x, long n, long stride, int bits,
                            uint16_t *s_out, uint16_t *z_out)
{
    double mn = INFINITY, mx = -INFINITY;
    for (long i = 0; i < n; ++i) {
        double v = orc_half_to_double(x[i * stride]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    int qmax = (1 << bits) - 1;
    uint16_t z = orc_double_to_half(mn, ORC_RD);
    uint16_t s = 0;
    if (mx > mn) {
        float zf = (float)orc_half_to_double(z);
        float mxf = (float)mx;
        float range = mxf - zf;
        float s32 = range / (float)qmax;
        s = orc_double_to_half((double)s32, ORC_RU);
        while (orc_half_to_double(z) + orc_half_to_double(s) * qmax < mx)
            s = half_next_up_positive(s);
    }
    *s_out = s;
    *z_out = z;
}

/* code = clamp(rint((x - z) / s), 0, 2^b - 1) in binary32; s == 0 gives 0. */
ORC_API int orc_affine_code(uint16_t x, uint16_t s, uint16_t z, int bits)
{
    if ((s & 0x7FFF) == 0)
        return 0;
    float xf = (float)orc_half_to_double(x);
    float zf = (float)orc_half_to_double(z);
    float sf = (float)orc_half_to_double(s);
    float d = xf - zf;
    float u = d / sf;
    float r = rintf(u);
    int qmax = (1 << bits) - 1;
    if (r < 0.0f) r = 0.0f;
    if (r > (float)qmax) r = (float)qmax;
    return (int)r;
}

/* Exact dequantized value code * s + z (binary64 is exact here). */
ORC_API double orc_affine_dequant(int code, uint16_t s, uint16_t z)
{
    return (double)code * orc_half_to_double(s) + orc_half_to_double(z);
}

/* ------------------------------------------------------------------ */
/* KIVI keys: per channel over groups of G tokens                       */
/* ------------------------------------------------------------------ */

/* x: fp16 [n_grp][G][D].  codes: uint8 [n_grp][G][D] (one code per byte).
 * sz: fp16 pairs [n_grp][D][2] = (scale, zero). */
ORC_API void orc_kivi_key_codes(int D, int G, int bits, const uint16_t *x, long n_grp,
                                uint8_t *codes, uint16_t *sz)
{
    for (long g = 0; g < n_grp; ++g) {
        const uint16_t *xg = x + g * (long)G * D;
        for (int c = 0; c < D; ++c) {
            uint16_t s, z;
            orc_affine_fit(xg + c, G, D, bits, &s, &z);
            sz[(g * D + c) * 2 + 0] = s;
            sz[(g * D + c) * 2 + 1] = z;
            for (int t = 0; t < G; ++t)
                codes[(g * G + t) * (long)D + c] = (uint8_t)orc_affine_code(xg[(long)t * D + c], s, z, bits);
        }
    }
}

/* Storage of a packed 2-bit KIVI key group (D = 128, G a multiple of 32).
 * The group is G/32 tiles of 1024 bytes.  Inside a tile, token t and
 * channel c are split as
 *   t = q + 8p        (q = t%8, p = (t%32)/8: the code sits in bits 2p)
 *   c = 16k + cc      (k = c/16), cc = 2r + e + 8h (r = (cc%8)/2, e = cc%2,
 *                                                    h = cc/8)
 * and the byte is number (e + 2h) of word k%4 in the 16-byte chunk
 * 4q + r of the 512-byte half k/4.  A byte therefore holds four tokens
 * q, q+8, q+16, q+24 of one channel, and the chunks 4q+r of both halves
 * hold tokens {q, q+8, q+16, q+24} x channels {16k+2r, 16k+2r+1, 16k+2r+8,
 * 16k+2r+9 : k = 0..7}: 32 contiguous bytes per (q, r). */
ORC_API long orc_kivi_key_byte_offset(int t, int c)
{
    long tile = t / 32;
    long q = t % 8;
    long k = c / 16, cc = c % 16;
    long r = (cc % 8) / 2, e = cc % 2, h = cc / 8;
    return tile * 1024 + (k / 4) * 512 + (4 * q + r) * 16 + (k % 4) * 4 + (e + 2 * h);
}

/* Bit position of token t inside its key byte. */
ORC_API int orc_kivi_key_bit(int t)
{
    return 2 * ((t % 32) / 8);
}

/* The same layout for b-bit codes (b = 2 or 4; KIVI-4 of the KIVI summary's
 * section 4): a byte holds 8/b codes, so a 32-token tile takes 1024 * b/2
 * bytes, made of b/2 planes of 1024 bytes.  Token t = q + 8p goes to plane
 * p / (8/b), at bits b * (p % (8/b)) of the byte that the 2-bit layout gives
 * inside the plane.  For b = 2 this is the layout above. */
ORC_API long orc_kivi_key_byte_offset_w(int bits, int t, int c)
{
    long cpb = 8 / bits;
    long p = (t % 32) / 8;
    return (t / 32) * (1024L * bits / 2) + (p / cpb) * 1024 + orc_kivi_key_byte_offset(t % 8, c);
}

ORC_API int orc_kivi_key_bit_w(int bits, int t)
{
    int cpb = 8 / bits;
    return bits * (((t % 32) / 8) % cpb);
}

ORC_API int orc_kivi_key_pack_w(int D, int G, int bits, const uint8_t *codes, long n_grp, uint8_t *packed)
{
    if (D != 128 || G % 32 != 0 || (bits != 2 && bits != 4))
        return 1;
    long gbytes = (long)G * D * bits / 8;
    int mask = (1 << bits) - 1;
    memset(packed, 0, (size_t)(gbytes * n_grp));
    for (long g = 0; g < n_grp; ++g)
        for (int t = 0; t < G; ++t)
            for (int c = 0; c < D; ++c) {
                int code = codes[(g * G + t) * (long)D + c] & mask;
                packed[g * gbytes + orc_kivi_key_byte_offset_w(bits, t, c)] |=
                    (uint8_t)(code << orc_kivi_key_bit_w(bits, t));
            }
    return 0;
}

ORC_API int orc_kivi_key_pack(int D, int G, const uint8_t *codes, long n_grp, uint8_t *packed)
{
    return orc_kivi_key_pack_w(D, G, 2, codes, n_grp, packed);
}

/* Storage index of channel c's scale (and, 128 entries later, its zero) in
 * a KIVI key group's parameter block of 128 fp16 scales followed by 128
 * fp16 zeros.  With c = 16k + 2r + e + 8h as for the codes, the entry is
 * number (k%2)*4 + e + 2h of the 8-entry chunk (k/2)*4 + r: chunk row r of
 * the codes finds its 32 channels in the chunks r, 4+r, 8+r, 12+r, in the
 * order of its code words. */
ORC_API int orc_kivi_key_sz_index(int c)
{
    int k = c / 16, cc = c % 16;
    int r = (cc % 8) / 2, e = cc % 2, h = cc / 8;
    return ((k / 2) * 4 + r) * 8 + (k % 2) * 4 + e + 2 * h;
}

/* sz: fp16 pairs [n_grp][D][2] -> stored blocks [n_grp][2*D]. */
ORC_API int orc_kivi_key_sz_pack(int D, const uint16_t *sz, long n_grp, uint16_t *stored)
{
    if (D != 128)
        return 1;
    for (long g = 0; g < n_grp; ++g)
        for (int c = 0; c < D; ++c) {
            stored[g * 2 * D + orc_kivi_key_sz_index(c)] = sz[(g * D + c) * 2 + 0];
            stored[g * 2 * D + D + orc_kivi_key_sz_index(c)] = sz[(g * D + c) * 2 + 1];
        }
    return 0;
}

static int kivi_key_code_at(int bits, const uint8_t *group_bytes, int t, int c)
{
    return (group_bytes[orc_kivi_key_byte_offset_w(bits, t, c)] >> orc_kivi_key_bit_w(bits, t)) & ((1 << bits) - 1);
}

/* ------------------------------------------------------------------ */
/* KIVI values: per token over groups of Gv channels                    */
/* ------------------------------------------------------------------ */

/* x: fp16 [n_tok][D].  codes [n_tok][D].  sz: fp16 pairs [n_tok][D/Gv][2]. */
ORC_API void orc_kivi_value_codes(int D, int Gv, int bits, const uint16_t *x, long n_tok,
                                  uint8_t *codes, uint16_t *sz)
{
    int ng = D / Gv;
    for (long t = 0; t < n_tok; ++t)
        for (int j = 0; j < ng; ++j) {
            uint16_t s, z;
            const uint16_t *xs = x + t * D + (long)j * Gv;
            orc_affine_fit(xs, Gv, 1, bits, &s, &z);
            sz[(t * ng + j) * 2 + 0] = s;
            sz[(t * ng + j) * 2 + 1] = z;
            for (int i = 0; i < Gv; ++i)
                codes[t * D + (long)j * Gv + i] = (uint8_t)orc_affine_code(xs[i], s, z, bits);
        }
}

/* Token-major b-bit packing (b = 2 or 4): byte c/(8/b) of the token's D*b/8
 * bytes, bits b*(c % (8/b)). */
ORC_API void orc_tokenmajor_pack_w(int D, int bits, const uint8_t *codes, long n_tok, uint8_t *packed)
{
    int cpb = 8 / bits, mask = (1 << bits) - 1;
    long tb = (long)D * bits / 8;
    memset(packed, 0, (size_t)(n_tok * tb));
    for (long t = 0; t < n_tok; ++t)
        for (int c = 0; c < D; ++c)
            packed[t * tb + c / cpb] |= (uint8_t)((codes[t * D + c] & mask) << (bits * (c % cpb)));
}

ORC_API void orc_tokenmajor_pack(int D, const uint8_t *codes, long n_tok, uint8_t *packed)
{
    orc_tokenmajor_pack_w(D, 2, codes, n_tok, packed);
}

/* KIVI value codes at 2 bits (D = 128) in value tiles: 32-token tiles of
 * 1024 bytes.  KIVI fixes the per-token grouping, not the storage order; this
 * order is a design choice (the fragment order of a tensor-core value product
 * whose rows are channels and whose k index runs over tokens), used by the
 * caches whose grouped-query heads decode on the tensor cores; the others keep
 * the token-major order (orc_tokenmajor_pack_w).  Token t, with
 * tt = t % 32 = 16 kv + 4 i + r (kv < 2, i < 4, r < 4), and channel
 * c = 32 g + 4 q + p (g < 4, q < 8, p < 4) sit at bits 2p of byte
 *   (t / 32) * 1024 + kv * 512 + (4q + r) * 16 + 4g + i,
 * so a byte holds four channels of one token, the 4-byte word 4q + r of a
 * 16-token half holds byte 8g + q of the tokens r, r + 4, r + 8, r + 12, and
 * the 16 bytes at (4q + r) * 16 are those words for g = 0..3. */
ORC_API long orc_kivi_value_byte_offset(int t, int c)
{
    int tt = t % 32, kv = tt / 16, i = (tt % 16) / 4, r = tt % 4;
    int g = c / 32, q = (c % 32) / 4;
    return (long)(t / 32) * 1024 + kv * 512 + (4 * q + r) * 16 + 4 * g + i;
}

ORC_API int orc_kivi_value_bit(int c) { return 2 * (c % 4); }

/* The 4-bit value tiles: 32-token tiles of 2048 bytes.  A byte holds channels
 * c and c + 64 (c < 64, low and high nibble) of one token.  With
 * t % 32 = 16 kv + 8 w + 4 s + r (kv, w, s < 2, r < 4) and
 * c % 64 = 16 m + 8 h + q (m < 4, h < 2, q < 8) the byte is
 *   (t / 32) * 2048 + kv * 1024 + (4q + r) * 32 + (2m + w) * 4 + 2h + s
 * and the nibble is c / 64: lane 4q + r's 32 bytes of a 16-token half are
 * eight words, word 2m + w holding channels 16m + q (bytes 0, 1) and
 * 16m + q + 8 (bytes 2, 3) of tokens r + 8w and r + 8w + 4 in its low nibbles
 * and channels 64 + 16m + q, 64 + 16m + q + 8 in its high nibbles. */
ORC_API long orc_kivi_value_byte_offset4(int t, int c)
{
    int tt = t % 32, kv = tt / 16, w = (tt / 8) % 2, s = (tt / 4) % 2, r = tt % 4;
    int c64 = c % 64, m = c64 / 16, h = (c64 / 8) % 2, q = c64 % 8;
    return (long)(t / 32) * 2048 + kv * 1024 + (4 * q + r) * 32 + (2 * m + w) * 4 + 2 * h + s;
}

ORC_API int orc_kivi_value_bit4(int c) { return 4 * (c / 64); }

/* Value codes [n_tok][D] -> packed bytes: with tiles the tile orders above
 * (ceil(n_tok / 32) tiles of 1024 or 2048 bytes; bytes of tokens past n_tok
 * stay 0), otherwise token-major (orc_tokenmajor_pack_w).  Returns 1 for
 * other shapes. */
ORC_API int orc_kivi_value_pack_w(int D, int bits, int tiles, const uint8_t *codes, long n_tok, uint8_t *packed)
{
    if (D != 128 || (bits != 2 && bits != 4))
        return 1;
    if (!tiles) {
        orc_tokenmajor_pack_w(D, bits, codes, n_tok, packed);
        return 0;
    }
    long tile = 16L * 32 * bits;
    memset(packed, 0, (size_t)((n_tok + 31) / 32 * tile));
    for (long t = 0; t < n_tok; ++t)
        for (int c = 0; c < D; ++c) {
            int code = codes[t * D + c] & ((1 << bits) - 1);
            if (bits == 2)
                packed[orc_kivi_value_byte_offset((int)(t % 32), c) + (t / 32) * tile] |=
                    (uint8_t)(code << orc_kivi_value_bit(c));
            else
                packed[orc_kivi_value_byte_offset4((int)(t % 32), c) + (t / 32) * tile] |=
                    (uint8_t)(code << orc_kivi_value_bit4(c));
        }
    return 0;
}

static int tokenmajor_code_at(int bits, const uint8_t *tok_bytes, int c);

static int kivi_value_code_at(int bits, int tiles, const uint8_t *vc, long t, int c)
{
    if (tiles && bits == 2)
        return (vc[(t / 32) * 1024 + orc_kivi_value_byte_offset((int)(t % 32), c)] >> orc_kivi_value_bit(c)) & 3;
    if (tiles)
        return (vc[(t / 32) * 2048 + orc_kivi_value_byte_offset4((int)(t % 32), c)] >> orc_kivi_value_bit4(c)) & 15;
    return tokenmajor_code_at(bits, vc + t * ((long)128 * bits / 8), c);
}

static int tokenmajor_code_at(int bits, const uint8_t *tok_bytes, int c)
{
    int cpb = 8 / bits;
    return (tok_bytes[c / cpb] >> (bits * (c % cpb))) & ((1 << bits) - 1);
}

/* ------------------------------------------------------------------ */
/* Kitty pages                                                          */
/* ------------------------------------------------------------------ */

/* Rows of the high plane: K rounded up to a multiple of 4 (rows K..Kp-1 hold
 * zero bytes), so that every 4-byte word of the plane belongs to one group of
 * four rows. */
ORC_API int orc_kitty_high_rows(int K) { return (K + 3) & ~3; }

ORC_API long orc_kitty_key_page_bytes(int D, int G, int K)
{
    return (long)D * G / 4 + (long)orc_kitty_high_rows(K) * G / 4 + D + 4L * D;
}

/* Storage order of the two code planes of a key page (D = 128, G a multiple
 * of 32).  The Kitty page (section "Page-Centric Memory Layout and
 * Dense-Sparse Decomposition") fixes which planes a page holds, not the order
 * of the bytes inside a plane; this one is a design choice.
 * Low plane: the page's low code bits (code & 3) of every channel in the
 * KIVI 2-bit key-tile order (orc_kivi_key_byte_offset): tile t/32 of 1024
 * bytes, token t % 32 = q + 8p of channel c = 16k + 2r + e + 8h at bits 2p
 * of byte (k/4)*512 + (4q + r)*16 + (k%4)*4 + e + 2h. */
ORC_API long orc_kitty_low_byte_offset(int t, int c) { return orc_kivi_key_byte_offset(t, c); }

/* High plane: the high code bits (code >> 2) of the boosted channels, row rho
 * = the rank of the channel among the boosted ones (ascending channel order).
 * Each 32-token tile owns a block of Kp * 8 bytes (Kp = orc_kitty_high_rows);
 * inside it, row rho = 16 kh + 4 r + b and token t % 32 = q + 8p sit at bits
 * 2p of byte kh*128 + 32 r + 4 q + b.  A 4-byte word thus holds four rows
 * 4r..4r+3 of a 16-row block at tokens q, q+8, q+16, q+24, and a partial last
 * block (Kp % 16 rows) is a compact prefix. */
ORC_API long orc_kitty_high_byte_offset(int K, int t, int rho)
{
    int kh = rho / 16, r = (rho % 16) / 4, b = rho % 4, q = (t % 32) % 8;
    return (long)(t / 32) * orc_kitty_high_rows(K) * 8 + kh * 128 + 32 * r + 4 * q + b;
}

/* Bit position of token t inside its byte, in both planes. */
ORC_API int orc_kitty_code_bit(int t) { return 2 * ((t % 32) / 8); }
ORC_API long orc_kitty_value_page_bytes(int D, int G) { return (long)G * D / 4 + 4L * G; }

/* Eq. 2 channel score, exactly: sum_t |x| in units of 2^-24 (every finite
 * fp16 is an integer multiple of 2^-24; 1/T is a common factor and does
 * not change the ranking). */
static int64_t kitty_abs_score(const uint16_t *x, int G, int D, int c)
{
    int64_t acc = 0;
    for (int t = 0; t < G; ++t)
        acc += (int64_t)ldexp(fabs(orc_half_to_double(x[(long)t * D + c])), 24);
    return acc;
}

/* Population variance over the page by sequential binary32 sums in token
 * order: var = sum(x^2)/T - (sum(x)/T)^2. */
static float kitty_var_score(const uint16_t *x, int G, int D, int c)
{
    float s1 = 0.0f, s2 = 0.0f;
    for (int t = 0; t < G; ++t) {
        float v = (float)orc_half_to_double(x[(long)t * D + c]);
        float sq = v * v;
        s1 = s1 + v;
        s2 = s2 + sq;
    }
    float T = (float)G;
    float m = s1 / T;
    float m2 = m * m;
    float e2 = s2 / T;
    return e2 - m2;
}

/* Top-K boost selection: K channels with the largest score, ties to the
 * lower channel index.  boosted[c] = 1 for the chosen channels. */
ORC_API void orc_kitty_select(int D, int G, int K, int score_mode, const uint16_t *x, uint8_t *boosted)
{
    int64_t *si = (int64_t *)malloc(sizeof(int64_t) * D);
    float *sf = (float *)malloc(sizeof(float) * D);
    for (int c = 0; c < D; ++c) {
        si[c] = kitty_abs_score(x, G, D, c);
        sf[c] = kitty_var_score(x, G, D, c);
        boosted[c] = 0;
    }
    for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int c = 0; c < D; ++c) {
            if (boosted[c])
                continue;
            if (best < 0) { best = c; continue; }
            int better = score_mode == 0 ? (si[c] > si[best]) : (sf[c] > sf[best]);
            if (better)
                best = c;
        }
        boosted[best] = 1;
    }
    free(si);
    free(sf);
}

/* Quantize one key page: x fp16 [G][D] -> packed record of
 * orc_kitty_key_page_bytes(D, G, K) bytes:
 *   low  D*G/4 bytes   code & 3 of every channel (orc_kitty_low_byte_offset)
 *   high Kp*G/4 bytes  code >> 2 of the r-th boosted channel (ascending order;
 *                      orc_kitty_high_byte_offset), Kp = K rounded up to 4
 *   idx  [D]           r for boosted channels, K + 1 otherwise
 *   s    fp16 [D], z fp16 [D]
 * Boosted channels use 4-bit codes, the rest 2-bit codes.  D = 128 and G a
 * multiple of 32 (the plane order); other shapes leave the page zero. */
ORC_API void orc_kitty_key_page(int D, int G, int K, int score_mode, const uint16_t *x, uint8_t *page)
{
    memset(page, 0, (size_t)orc_kitty_key_page_bytes(D, G, K));
    if (D != 128 || G % 32 != 0)
        return;
    uint8_t *boosted = (uint8_t *)malloc((size_t)D);
    orc_kitty_select(D, G, K, score_mode, x, boosted);
    uint8_t *low = page;
    uint8_t *high = page + (long)D * G / 4;
    uint8_t *idx = high + (long)orc_kitty_high_rows(K) * G / 4;
    uint16_t *s = (uint16_t *)(idx + D);
    uint16_t *z = s + D;
    int r = 0;
    for (int c = 0; c < D; ++c) {
        int bits = boosted[c] ? 4 : 2;
        orc_affine_fit(x + c, G, D, bits, &s[c], &z[c]);
        idx[c] = boosted[c] ? (uint8_t)r : (uint8_t)(K + 1);
        for (int t = 0; t < G; ++t) {
            int code = orc_affine_code(x[(long)t * D + c], s[c], z[c], bits);
            low[orc_kitty_low_byte_offset(t, c)] |= (uint8_t)((code & 3) << orc_kitty_code_bit(t));
            if (boosted[c])
                high[orc_kitty_high_byte_offset(K, t, r)] |= (uint8_t)(((code >> 2) & 3) << orc_kitty_code_bit(t));
        }
        if (boosted[c])
            ++r;
    }
    free(boosted);
}

/* Algorithm 1 reconstruction of the integer codes of a key page:
 * X = low | (high << 2) with high taken from row idx[c] when idx[c] < K
 * (and implicitly 0 otherwise).  codes [G][D], s [D], z [D]. */
ORC_API void orc_kitty_key_page_decode(int D, int G, int K, const uint8_t *page,
                                       uint8_t *codes, uint16_t *s_out, uint16_t *z_out)
{
    if (D != 128 || G % 32 != 0)
        return;
    const uint8_t *low = page;
    const uint8_t *high = page + (long)D * G / 4;
    const uint8_t *idx = high + (long)orc_kitty_high_rows(K) * G / 4;
    const uint16_t *s = (const uint16_t *)(idx + D);
    const uint16_t *z = s + D;
    for (int c = 0; c < D; ++c) {
        s_out[c] = s[c];
        z_out[c] = z[c];
        for (int t = 0; t < G; ++t) {
            int lo = (low[orc_kitty_low_byte_offset(t, c)] >> orc_kitty_code_bit(t)) & 3;
            int hi = 0;
            if (idx[c] < K)
                hi = (high[orc_kitty_high_byte_offset(K, t, idx[c])] >> orc_kitty_code_bit(t)) & 3;
            codes[(long)t * D + c] = (uint8_t)(lo | (hi << 2));
        }
    }
}

/* Value page: per token over all D channels, 2-bit.  x fp16 [G][D] ->
 * codes [G][D/4] (token-major packing), s fp16 [G], z fp16 [G]. */
ORC_API void orc_kitty_value_page(int D, int G, const uint16_t *x, uint8_t *page)
{
    uint8_t *codes = (uint8_t *)malloc((size_t)G * D);
    uint16_t *sz = (uint16_t *)malloc(sizeof(uint16_t) * 2 * G);
    orc_kivi_value_codes(D, D, 2, x, G, codes, sz);
    orc_tokenmajor_pack(D, codes, G, page);
    uint16_t *s = (uint16_t *)(page + (long)G * D / 4);
    uint16_t *z = s + G;
    for (int t = 0; t < G; ++t) {
        s[t] = sz[2 * t];
        z[t] = sz[2 * t + 1];
    }
    free(codes);
    free(sz);
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 and the WitCert dither                                 */
/* ------------------------------------------------------------------ */

/* One Philox4x32 round: two 32x32->64 products, a Feistel-like swap. */
static void philox_round(uint32_t x[4], const uint32_t k[2])
{
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)x[0];
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)x[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t y0 = hi1 ^ x[1] ^ k[0];
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x[3] ^ k[1];
    uint32_t y3 = lo0;
    x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
}

ORC_API void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t x[4] = { ctr[0], ctr[1], ctr[2], ctr[3] };
    uint32_t k[2] = { key[0], key[1] };
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k[0] += 0x9E3779B9u;   /* golden ratio */
            k[1] += 0xBB67AE85u;   /* sqrt(3) - 1 */
        }
        philox_round(x, k);
    }
    memcpy(out, x, sizeof(x));
}

/* Inverse of the ten rounds (used only to pin the forward map). */
ORC_API void orc_philox4x32_10_inverse(const uint32_t out[4], const uint32_t key[2], uint32_t ctr[4])
{
    uint32_t x[4] = { out[0], out[1], out[2], out[3] };
    for (int r = 9; r >= 0; --r) {
        uint32_t k0 = key[0] + 0x9E3779B9u * (uint32_t)r;
        uint32_t k1 = key[1] + 0xBB67AE85u * (uint32_t)r;
        /* forward: y1 = lo(M1*x2), y3 = lo(M0*x0); both multipliers are odd,
         * so they are invertible mod 2^32 (Newton: x <- x(2 - a x)). */
        uint32_t inv0 = 0xD2511F53u, inv1 = 0xCD9E8D57u;
        for (int i = 0; i < 5; ++i) { inv0 *= 2u - 0xD2511F53u * inv0; inv1 *= 2u - 0xCD9E8D57u * inv1; }
        uint32_t x0 = x[3] * inv0;
        uint32_t x2 = x[1] * inv1;
        uint64_t p0 = (uint64_t)0xD2511F53u * x0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
        uint32_t x1 = x[0] ^ (uint32_t)(p1 >> 32) ^ k0;
        uint32_t x3 = x[2] ^ (uint32_t)(p0 >> 32) ^ k1;
        x[0] = x0; x[1] = x1; x[2] = x2; x[3] = x3;
    }
    memcpy(ctr, x, sizeof(x));
}

/* Dither xi in [-1/2, 1/2) for one element.  Counter = (token, channel/4,
 * (layer << 17) | (kv_sel << 16) | kv_head, request); key = (seed low
 * word, seed high word); the channel selects output word channel % 4;
 * xi = (word >> 8) * 2^-24 - 1/2 (exact in binary32). */
ORC_API float orc_dither(uint64_t seed, int32_t request, int32_t layer, int kv_sel,
                         int32_t kv_head, int32_t token, int32_t channel)
{
    uint32_t ctr[4], key[2], out[4];
    ctr[0] = (uint32_t)token;
    ctr[1] = (uint32_t)channel >> 2;
    ctr[2] = ((uint32_t)layer << 17) | ((uint32_t)(kv_sel & 1) << 16) | ((uint32_t)kv_head & 0xFFFFu);
    ctr[3] = (uint32_t)request;
    key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    key[1] = (uint32_t)(seed >> 32);
    orc_philox4x32_10(ctr, key, out);
    float u = (float)(out[channel & 3] >> 8) * 0x1.0p-24f;
    return u - 0.5f;
}

/* Quantize one block of T tokens (T = 256 in the method) of one (request,
 * kv head): x fp16 [T][D].  s_c = fp16_RN(amax_c / 126.5) with binary32
 * division; code = clamp(rint(x/s + xi), -127, 127) in binary32 using the
 * stored fp16 scale; s == 0 gives code 0.  codes int8 [T][D], scale fp16 [D]. */
ORC_API void orc_int8_quant_block(int D, int T, const uint16_t *x, uint64_t seed, int32_t request,
                                  int32_t layer, int kv_sel, int32_t kv_head, int32_t tok0,
                                  int8_t *codes, uint16_t *scale)
{
    for (int c = 0; c < D; ++c) {
        double amax = 0.0;
        for (int t = 0; t < T; ++t) {
            double v = fabs(orc_half_to_double(x[(long)t * D + c]));
            if (v > amax) amax = v;
        }
        float s32 = (float)amax / 126.5f;
        uint16_t s = orc_double_to_half((double)s32, ORC_RN);
        scale[c] = s;
        float sf = (float)orc_half_to_double(s);
        for (int t = 0; t < T; ++t) {
            int code = 0;
            if (sf != 0.0f) {
                float xf = (float)orc_half_to_double(x[(long)t * D + c]);
                float xi = orc_dither(seed, request, layer, kv_sel, kv_head, tok0 + t, c);
                float u = xf / sf;
                float w = u + xi;
                float r = rintf(w);
                if (r < -127.0f) r = -127.0f;
                if (r > 127.0f) r = 127.0f;
                code = (int)r;
            }
            codes[(long)t * D + c] = (int8_t)code;
        }
    }
}

/* Dequantized value s * (code - xi), exactly in binary64. */
ORC_API double orc_int8_dequant(int code, uint16_t s, float xi)
{
    return orc_half_to_double(s) * ((double)code - (double)xi);
}

/* ------------------------------------------------------------------ */
/* Attention in binary64 (no splitting)                                 */
/* ------------------------------------------------------------------ */

/* softmax(sm_scale * q.K^T) V over n tokens; k, v binary64 [n][D]. */
static void attend_f64(int D, int n, const double *q, const double *k, const double *v,
                       double sm_scale, double *out)
{
    double *sc = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        double a = 0.0;
        for (int c = 0; c < D; ++c)
            a += q[c] * k[(long)t * D + c];
        sc[t] = sm_scale * a;
        if (sc[t] > m) m = sc[t];
    }
    double l = 0.0;
    for (int t = 0; t < n; ++t) {
        sc[t] = exp(sc[t] - m);
        l += sc[t];
    }
    for (int c = 0; c < D; ++c)
        out[c] = 0.0;
    for (int t = 0; t < n; ++t) {
        double p = sc[t] / l;
        for (int c = 0; c < D; ++c)
            out[c] += p * v[(long)t * D + c];
    }
    free(sc);
}

/* Textbook attention of fp16 inputs (used to pin the residual-only case). */
ORC_API void orc_attend_fp16(int D, int n, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             double sm_scale, double *out)
{
    double *qd = (double *)malloc(sizeof(double) * D);
    double *kd = (double *)malloc(sizeof(double) * (size_t)n * D + 8);
    double *vd = (double *)malloc(sizeof(double) * (size_t)n * D + 8);
    for (int c = 0; c < D; ++c) qd[c] = orc_half_to_double(q[c]);
    for (long i = 0; i < (long)n * D; ++i) {
        kd[i] = orc_half_to_double(k[i]);
        vd[i] = orc_half_to_double(v[i]);
    }
    attend_f64(D, n, qd, kd, vd, sm_scale, out);
    free(qd); free(kd); free(vd);
}

/* KIVI cache of one (batch row, kv head) at attention time with L tokens:
 *   key residual holds r_K = ((L-1) mod R) + 1 tokens, the first L - r_K
 *   keys are quantized in groups of G; value residual holds min(L, R)
 *   tokens, the first L - min(L, R) values are quantized per token.
 *   Residual token t lives at slot t % R.
 * Arrays (this (b, kvh) only), b_K / b_V-bit codes:
 *   kc   packed key groups, G*D*b_K/8 bytes each   ksz fp16 [grp][D][2]
 *   vc   packed value codes (orc_kivi_value_pack_w: value tiles when
 *        vtiles, else token-major)                vsz fp16 [tok][D/Gv][2]
 *   kres, vres fp16 [R][D]
 * out: binary64 [g][D] for the g query heads q fp16 [g][D]. */
ORC_API void orc_kivi_decode_one_w(int D, int G, int Gv, int R, int L, int bits_k, int bits_v, int vtiles, int n_heads,
                                   double sm_scale, const uint16_t *q, const uint8_t *kc, const uint16_t *ksz,
                                   const uint8_t *vc, const uint16_t *vsz,
                                   const uint16_t *kres, const uint16_t *vres, double *out)
{
    int rK = ((L - 1) % R) + 1;
    int nKq = L - rK;
    int rV = L < R ? L : R;
    int nVq = L - rV;
    int ngv = D / Gv;
    double *k = (double *)malloc(sizeof(double) * (size_t)L * D);
    double *v = (double *)malloc(sizeof(double) * (size_t)L * D);
    for (int t = 0; t < L; ++t) {
        for (int c = 0; c < D; ++c) {
            if (t < nKq) {
                long g = t / G;
                const uint8_t *gb = kc + g * ((long)G * D * bits_k / 8);
                int code = kivi_key_code_at(bits_k, gb, t % G, c);
                k[(long)t * D + c] = orc_affine_dequant(code, ksz[(g * D + c) * 2], ksz[(g * D + c) * 2 + 1]);
            } else {
                k[(long)t * D + c] = orc_half_to_double(kres[(long)(t % R) * D + c]);
            }
            if (t < nVq) {
                int code = kivi_value_code_at(bits_v, vtiles, vc, t, c);
                long j = (long)t * ngv + c / Gv;
                v[(long)t * D + c] = orc_affine_dequant(code, vsz[j * 2], vsz[j * 2 + 1]);
            } else {
                v[(long)t * D + c] = orc_half_to_double(vres[(long)(t % R) * D + c]);
            }
        }
    }
    double *qd = (double *)malloc(sizeof(double) * D);
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < D; ++c) qd[c] = orc_half_to_double(q[(long)h * D + c]);
        attend_f64(D, L, qd, k, v, sm_scale, out + (long)h * D);
    }
    free(qd); free(k); free(v);
}

ORC_API void orc_kivi_decode_one(int D, int G, int Gv, int R, int L, int n_heads, double sm_scale,
                                 const uint16_t *q, const uint8_t *kc, const uint16_t *ksz,
                                 const uint8_t *vc, const uint16_t *vsz,
                                 const uint16_t *kres, const uint16_t *vres, double *out)
{
    orc_kivi_decode_one_w(D, G, Gv, R, L, 2, 2, 0, n_heads, sm_scale, q, kc, ksz, vc, vsz, kres, vres, out);
}

/* Kitty cache of one (batch row, kv head) with L tokens, sink S, page G,
 * value local window R:
 *   keys:   sink [0, min(L,S)); pages; key Q-buffer of
 *           n_kb = ((L-S-1) mod G) + 1 tokens (L > S), slot (t-S) % G.
 *   values: sink; pages; value Q-buffer of n_vb = ((E-1) mod G) + 1 tokens
 *           (E = L-S-R evicted tokens, E > 0), slot (t-S) % G; local window
 *           of the last min(L-S, R) tokens, slot t % R.
 * kp / vp: consecutive key / value page records. */
ORC_API void orc_kitty_decode_one(int D, int G, int K, int S, int R, int L, int n_heads, double sm_scale,
                                  const uint16_t *q, const uint8_t *kp, const uint8_t *vp,
                                  const uint16_t *ksink, const uint16_t *vsink,
                                  const uint16_t *kqbuf, const uint16_t *vqbuf, const uint16_t *vlocal,
                                  double *out)
{
    int nkb = L > S ? ((L - S - 1) % G) + 1 : 0;
    int PK = L > S ? (L - S - nkb) / G : 0;
    int E = L - S - R; if (E < 0) E = 0;
    int nvb = E > 0 ? ((E - 1) % G) + 1 : 0;
    int PV = (E - nvb) / G;
    long kpb = orc_kitty_key_page_bytes(D, G, K);
    long vpb = orc_kitty_value_page_bytes(D, G);
    double *k = (double *)malloc(sizeof(double) * (size_t)L * D);
    double *v = (double *)malloc(sizeof(double) * (size_t)L * D);
    uint8_t *codes = (uint8_t *)malloc((size_t)G * D);
    uint16_t *s = (uint16_t *)malloc(sizeof(uint16_t) * D);
    uint16_t *z = (uint16_t *)malloc(sizeof(uint16_t) * D);
    for (int t = 0; t < L; ++t) {
        if (t < S) {
            for (int c = 0; c < D; ++c) k[(long)t * D + c] = orc_half_to_double(ksink[(long)t * D + c]);
        } else if (t < S + PK * G) {
            /* filled page by page below */
        } else {
            int slot = (t - S) % G;
            for (int c = 0; c < D; ++c) k[(long)t * D + c] = orc_half_to_double(kqbuf[(long)slot * D + c]);
        }
    }
    for (int p = 0; p < PK; ++p) {
        orc_kitty_key_page_decode(D, G, K, kp + p * kpb, codes, s, z);
        for (int tt = 0; tt < G; ++tt)
            for (int c = 0; c < D; ++c)
                k[(long)(S + p * G + tt) * D + c] = orc_affine_dequant(codes[(long)tt * D + c], s[c], z[c]);
    }
    for (int t = 0; t < L; ++t) {
        for (int c = 0; c < D; ++c) {
            double val;
            if (t < S) {
                val = orc_half_to_double(vsink[(long)t * D + c]);
            } else if (t < S + PV * G) {
                int p = (t - S) / G, tt = (t - S) % G;
                const uint8_t *pg = vp + p * vpb;
                const uint16_t *ps = (const uint16_t *)(pg + (long)G * D / 4);
                int code = tokenmajor_code_at(2, pg + (long)tt * (D / 4), c);
                val = orc_affine_dequant(code, ps[tt], ps[G + tt]);
            } else if (t < S + PV * G + nvb) {
                val = orc_half_to_double(vqbuf[(long)((t - S) % G) * D + c]);
            } else {
                val = orc_half_to_double(vlocal[(long)(t % R) * D + c]);
            }
            v[(long)t * D + c] = val;
        }
    }
    double *qd = (double *)malloc(sizeof(double) * D);
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < D; ++c) qd[c] = orc_half_to_double(q[(long)h * D + c]);
        attend_f64(D, L, qd, k, v, sm_scale, out + (long)h * D);
    }
    free(qd); free(k); free(v); free(codes); free(s); free(z);
}

/* INT8 dithered cache of one (batch row = request, kv head) with L tokens
 * and blocks of T tokens: the first L - n_tail tokens are quantized, with
 * n_tail = ((L-1) mod T) + 1 fp16 tokens in the active block (slot t % T).
 * kc, vc int8 [L][D]; ks, vs fp16 [blocks][D]; ktail, vtail fp16 [T][D]. */
ORC_API void orc_int8_decode_one(int D, int T, int L, int n_heads, double sm_scale,
                                 uint64_t seed, int32_t request, int32_t layer, int32_t kv_head,
                                 const uint16_t *q, const int8_t *kc, const int8_t *vc,
                                 const uint16_t *ks, const uint16_t *vs,
                                 const uint16_t *ktail, const uint16_t *vtail, double *out)
{
    int ntail = ((L - 1) % T) + 1;
    int nq = L - ntail;
    double *k = (double *)malloc(sizeof(double) * (size_t)L * D);
    double *v = (double *)malloc(sizeof(double) * (size_t)L * D);
    for (int t = 0; t < L; ++t)
        for (int c = 0; c < D; ++c) {
            if (t < nq) {
                long blk = t / T;
                float xk = orc_dither(seed, request, layer, 0, kv_head, t, c);
                float xv = orc_dither(seed, request, layer, 1, kv_head, t, c);
                k[(long)t * D + c] = orc_int8_dequant(kc[(long)t * D + c], ks[blk * D + c], xk);
                v[(long)t * D + c] = orc_int8_dequant(vc[(long)t * D + c], vs[blk * D + c], xv);
            } else {
                k[(long)t * D + c] = orc_half_to_double(ktail[(long)(t % T) * D + c]);
                v[(long)t * D + c] = orc_half_to_double(vtail[(long)(t % T) * D + c]);
            }
        }
    double *qd = (double *)malloc(sizeof(double) * D);
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < D; ++c) qd[c] = orc_half_to_double(q[(long)h * D + c]);
        attend_f64(D, L, qd, k, v, sm_scale, out + (long)h * D);
    }
    free(qd); free(k); free(v);
}

/* ------------------------------------------------------------------ */
/* Token-granular INT8 over a slot pool (WitCert, SGLang storage)        */
/* ------------------------------------------------------------------ */

/* Dither of the slot-keyed stream.  The tuple is (layer, KV head, slot,
 * channel); counter = (slot, channel/4, (layer << 17) | (kv_sel << 16) |
 * kv_head, 0), key and output word as orc_dither. */
ORC_API float orc_dither_slot(uint64_t seed, int32_t layer, int kv_sel, int32_t kv_head, int32_t slot,
                              int32_t channel)
{
    uint32_t ctr[4], key[2], out[4];
    ctr[0] = (uint32_t)slot;
    ctr[1] = (uint32_t)channel >> 2;
    ctr[2] = ((uint32_t)layer << 17) | ((uint32_t)(kv_sel & 1) << 16) | ((uint32_t)kv_head & 0xFFFFu);
    ctr[3] = 0u;
    key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
    key[1] = (uint32_t)(seed >> 32);
    orc_philox4x32_10(ctr, key, out);
    float u = (float)(out[channel & 3] >> 8) * 0x1.0p-24f;
    return u - 0.5f;
}

/* Quantize one token of one kv head written to `slot`: x fp16 [D].  For
 * every group of Gc consecutive channels s = fp16_RN(amax / 126.5) (binary32
 * division); code = clamp(rint(x/s + xi), -127, 127) in binary32 with the
 * stored scale; s == 0 gives code 0.  codes int8 [D], scale fp16 [D/Gc]. */
ORC_API void orc_int8t_quant_token(int D, int Gc, const uint16_t *x, uint64_t seed, int32_t layer, int kv_sel,
                                   int32_t kv_head, int32_t slot, int8_t *codes, uint16_t *scale)
{
    for (int g = 0; g < D / Gc; ++g) {
        double amax = 0.0;
        for (int i = 0; i < Gc; ++i) {
            double v = fabs(orc_half_to_double(x[g * Gc + i]));
            if (v > amax) amax = v;
        }
        float s32 = (float)amax / 126.5f;
        uint16_t s = orc_double_to_half((double)s32, ORC_RN);
        scale[g] = s;
        float sf = (float)orc_half_to_double(s);
        for (int i = 0; i < Gc; ++i) {
            int c = g * Gc + i;
            int code = 0;
            if (sf != 0.0f) {
                float xf = (float)orc_half_to_double(x[c]);
                float xi = orc_dither_slot(seed, layer, kv_sel, kv_head, slot, c);
                float u = xf / sf;
                float w = u + xi;
                float r = rintf(w);
                if (r < -127.0f) r = -127.0f;
                if (r > 127.0f) r = 127.0f;
                code = (int)r;
            }
            codes[c] = (int8_t)code;
        }
    }
}

/* Decode of one (request, kv head) over a slot pool: token t of the request
 * lives in slot table[t]; kc, vc int8 [n_slots][Hkv][D]; ks, vs fp16
 * [n_slots][Hkv][D/Gc].  Every token is dequantized as s (code - xi) with the
 * dither of its slot, then softmax attention in binary64 over the L tokens. */
ORC_API void orc_int8t_decode_one(int D, int Gc, int Hkv, int L, int n_heads, double sm_scale, uint64_t seed,
                                  int32_t layer, int32_t kv_head, const int32_t *table, const uint16_t *q,
                                  const int8_t *kc, const int8_t *vc, const uint16_t *ks, const uint16_t *vs,
                                  double *out)
{
    double *k = (double *)malloc(sizeof(double) * (size_t)L * D + 8);
    double *v = (double *)malloc(sizeof(double) * (size_t)L * D + 8);
    for (int t = 0; t < L; ++t) {
        long rec = (long)table[t] * Hkv + kv_head;
        for (int c = 0; c < D; ++c) {
            float xk = orc_dither_slot(seed, layer, 0, kv_head, table[t], c);
            float xv = orc_dither_slot(seed, layer, 1, kv_head, table[t], c);
            k[(long)t * D + c] = orc_int8_dequant(kc[rec * D + c], ks[rec * (D / Gc) + c / Gc], xk);
            v[(long)t * D + c] = orc_int8_dequant(vc[rec * D + c], vs[rec * (D / Gc) + c / Gc], xv);
        }
    }
    double *qd = (double *)malloc(sizeof(double) * D);
    for (int h = 0; h < n_heads; ++h) {
        for (int c = 0; c < D; ++c) qd[c] = orc_half_to_double(q[(long)h * D + c]);
        attend_f64(D, L, qd, k, v, sm_scale, out + (long)h * D);
    }
    free(qd); free(k); free(v);
}
