// Write-side kernels: KIVI key groups and value tokens, Kitty key / value
// pages, WitCert INT8 subtractive dither, and the Philox diagnostic.
//
// Bit-exactness: every fp32 operation that decides a code is an explicit
// round-to-nearest intrinsic (__fsub_rn, __fdiv_rn, rintf) so that no FMA
// contraction or approximate division changes a code; scales and zeros are
// rounded with the directed fp16 conversions the C ABI documents.
#include "kvq_device.cuh"
#include "kvq_quant.cuh"
#include "kvq_internal.h"

namespace kvq {

// ---------------------------------------------------------------------------
// a1: KIVI key groups.  One CTA (4 warps) per group of G = 32*NT tokens;
// warp w owns channels [32w, 32w+32); lane t holds token t of every 32-token
// tile.  Per-channel min / max is a warp-shuffle reduce-scatter that leaves
// lane l with channel 32w + l; codes are packed in registers, OR-reduced
// across the four lanes t, t^8, t^16, t^24 that share a byte, and stored as
// 8-byte pieces of the tile layout (KIVI section 3.3; Kitty Observation 1
// formula).  Tile layout: token t = q + 8p, channel c = 16k + 2r + e + 8h
// sits in bits 2p of byte e + 2h of word k%4 of chunk 4q + r of half k/4.
// The (s, z) block of a group is 128 fp16 scales then 128 fp16 zeros, both
// at ((k/2)*4 + r)*8 + (k%2)*4 + e + 2h.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int kivi_sz_index(int c) {
    const int k = c >> 4, cc = c & 15;
    return ((k >> 1) * 4 + ((cc & 7) >> 1)) * 8 + (k & 1) * 4 + (cc & 1) + 2 * (cc >> 3);
}

// One key group by a 128-thread block: src fp16 [G][D], codes the group's
// G*D*bits/8 bytes, sz the group's 2*D fp16 (scales, then zeros).  bits = 2
// or 4: a 32-token tile is bits/2 planes of 1024 bytes, token q + 8p in plane
// p / (8/bits) at bits bits*(p % (8/bits)) of its 2-bit-layout byte.
// One key group by a 128-thread block, thread c = channel c: src fp16 [G][D],
// codes the group's G*D*BITS/8 bytes, sz the group's 2*D fp16 (scales, then
// zeros).  The group is staged in shared memory (xs) with 16-byte loads; each
// thread reads its channel's column (min / max, fit, codes) and writes its
// code bytes into a shared copy of the tile layout (cw), which the block then
// stores with 16-byte stores.  BITS = 2 or 4: a 32-token tile is BITS/2
// planes of 1024 bytes, token q + 8p in plane p / (8/BITS) at bits
// BITS*(p % (8/BITS)) of its 2-bit-layout byte.  Every thread of the block
// calls it (block barriers inside).
// The codes of the thread's channel over the group staged in xs, as bytes of
// the tile layout in cb (product form, or the quotient when EXACT); returns
// whether the product form met a near-tie.
template <int NT, int BITS, bool EXACT>
__device__ __forceinline__ bool key_group_codes(const uint16_t *xs, uint8_t *cb, int c, int pos, float zf, float sf,
                                                float rf) {
    constexpr int CPB = 8 / BITS, NPL = BITS / 2, QMAX = (1 << BITS) - 1;
    bool tie = false;
#pragma unroll
    for (int tt = 0; tt < NT; ++tt)
#pragma unroll 2
        for (int q = 0; q < 8; ++q) {
            uint32_t byte[NPL];
#pragma unroll
            for (int pl = 0; pl < NPL; ++pl) byte[pl] = 0u;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float x = h2f(xs[(tt * 32 + q + 8 * p) * KVQ_D + c]);
                const uint32_t code = EXACT ? (uint32_t)affine_code(x, zf, sf, rf, QMAX)
                                            : (uint32_t)affine_code_fast(x, zf, rf, tie);
                byte[p / CPB] |= code << (BITS * (p % CPB));
            }
#pragma unroll
            for (int pl = 0; pl < NPL; ++pl) cb[(tt * NPL + pl) * 1024 + q * 64 + pos] = (uint8_t)byte[pl];
        }
    return tie;
}

// One key group staged in xs (visible to the whole block) by a 128-thread
// block, thread c = channel c: codes the group's G*D*BITS/8 bytes, sz its
// 2*D fp16 (scales, then zeros).  Each thread reads its channel's column
// (min / max, fit, codes) and writes its code bytes into a shared copy of
// the tile layout (cw), which the block then stores with 16-byte stores.
// BITS = 2 or 4: a 32-token tile is BITS/2 planes of 1024 bytes, token
// q + 8p in plane p / (8/BITS) at bits BITS*(p % (8/BITS)) of its
// 2-bit-layout byte.  Every thread of the block calls it (a block barrier
// inside; cw is read by the block until its next barrier).
template <int NT, int BITS>
__device__ __forceinline__ void key_group_code_b(const uint16_t *xs, uint8_t *__restrict__ codes,
                                                 uint16_t *__restrict__ sz, uint32_t *cw) {
    constexpr int G = 32 * NT, NPL = BITS / 2, QMAX = (1 << BITS) - 1;
    const int c = threadIdx.x;
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll 8
    for (int t = 0; t < G; ++t) {
        const float v = h2f(xs[t * KVQ_D + c]);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    uint16_t s, z;
    affine_fit(mn, mx, QMAX, s, z);
    const int si = kivi_sz_index(c);
    sz[si] = s;
    sz[KVQ_D + si] = z;
    const float sf = h2f(s), zf = h2f(z), rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
    // channel c = 16k + 2r + e + 8h: half k/4, chunk row 4q + r, word k%4, byte e + 2h of the tile layout
    const int k = c >> 4, cc = c & 15;
    const int pos = (k >> 2) * 512 + ((cc & 7) >> 1) * 16 + (k & 3) * 4 + (cc & 1) + 2 * (cc >> 3);
    uint8_t *cb = reinterpret_cast<uint8_t *>(cw);
    // the product form; a thread that met a near-tie redoes its column with the quotient
    if (key_group_codes<NT, BITS, false>(xs, cb, c, pos, zf, sf, rf))
        key_group_codes<NT, BITS, true>(xs, cb, c, pos, zf, sf, rf);
    __syncthreads();
    const uint4 *c4 = reinterpret_cast<const uint4 *>(cw);
    uint4 *o4 = reinterpret_cast<uint4 *>(codes);
#pragma unroll
    for (int i = c; i < NT * NPL * 64; i += 128) o4[i] = c4[i];
}

// One key group from global memory: staged with 16-byte loads, then coded.
template <int NT, int BITS>
__device__ __forceinline__ void key_group_quant_b(const uint16_t *__restrict__ src, uint8_t *__restrict__ codes,
                                                  uint16_t *__restrict__ sz, uint16_t *xs, uint32_t *cw) {
    const int c = threadIdx.x;
    __syncthreads();                                               // the block's previous group is stored
    {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *x4 = reinterpret_cast<uint4 *>(xs);
#pragma unroll
        for (int i = 0; i < 4 * NT; ++i) x4[c + 128 * i] = __ldg(s4 + c + 128 * i);
    }
    __syncthreads();
    key_group_code_b<NT, BITS>(xs, codes, sz, cw);
}

template <int NT>
__device__ __forceinline__ void key_group_quant(const uint16_t *__restrict__ src, uint8_t *__restrict__ codes,
                                                uint16_t *__restrict__ sz, int bits = 2) {
    __shared__ __align__(16) uint16_t xs[32 * NT * KVQ_D];
    __shared__ __align__(16) uint32_t cw[NT * 2 * 256];           // NT tiles x up to 2 planes x 1024 bytes
    if (bits == 4) key_group_quant_b<NT, 4>(src, codes, sz, xs, cw);
    else key_group_quant_b<NT, 2>(src, codes, sz, xs, cw);
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Bulk key groups: a grid of resident blocks walks the groups; with G <= 64
// each block copies its next group (cp.async) into a second buffer while it
// codes the current one.
template <int NT, int BITS>
__global__ void __launch_bounds__(128) quant_key_kivi_kernel(const uint16_t *__restrict__ k, int64_t n_groups,
                                                             uint8_t *__restrict__ codes, uint16_t *__restrict__ sz) {
    constexpr int G = 32 * NT;
    int64_t g = blockIdx.x;
    if (g >= n_groups) return;
    if constexpr (NT <= 2) {
        __shared__ __align__(16) uint16_t xs[2][G * KVQ_D];
        __shared__ __align__(16) uint32_t cw[NT * 2 * 256];
        const int c = threadIdx.x;
        auto issue = [&](int64_t gg, int b) {
            const uint4 *src = reinterpret_cast<const uint4 *>(k + gg * (int64_t)G * KVQ_D);
            uint4 *dst = reinterpret_cast<uint4 *>(xs[b]);
#pragma unroll
            for (int i = 0; i < 4 * NT; ++i) cp_async16(dst + c + 128 * i, src + c + 128 * i);
        };
        issue(g, 0);
        cp_async_commit();
        for (int b = 0; g < n_groups; g += gridDim.x, b ^= 1) {
            if (g + gridDim.x < n_groups) issue(g + gridDim.x, b ^ 1);
            cp_async_commit();                                     // (an empty group past the end)
            cp_async_wait_prev();                                  // this thread's copies of group g are in
            __syncthreads();                                       // and every thread's; cw free again
            key_group_code_b<NT, BITS>(xs[b], codes + g * (int64_t)G * KVQ_D * BITS / 8, sz + g * 2 * KVQ_D, cw);
        }
    } else {
        for (; g < n_groups; g += gridDim.x)
            key_group_quant<NT>(k + g * (int64_t)G * KVQ_D, codes + g * (int64_t)G * KVQ_D * BITS / 8,
                                sz + g * 2 * KVQ_D, BITS);
    }
}

// One value token by a warp, per token over groups of GV channels: lane l
// reads channels 4l..4l+3 and returns in wv the packed word of its lane quad
// (valid in lanes 4j, channels 16j..16j+15) and the (s, z) of its group.
template <int GV>
__device__ __forceinline__ void value_token_quant_x(uint2 u, int lane, uint32_t &wv, uint16_t &s, uint16_t &z,
                                                    int bits = 2) {
    constexpr int LG = GV / 4;   // lanes per group
    float x0 = h2f(lo16(u.x)), x1 = h2f(hi16(u.x)), x2 = h2f(lo16(u.y)), x3 = h2f(hi16(u.y));
    float mn = fminf(fminf(x0, x1), fminf(x2, x3));
    float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
#pragma unroll
    for (int o = 1; o < LG; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    const int qmax = (1 << bits) - 1;
    affine_fit(mn, mx, qmax, s, z);
    const float sf = h2f(s), zf = h2f(z), rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
    const uint32_t b = (uint32_t)affine_code(x0, zf, sf, rf, qmax) |
                       ((uint32_t)affine_code(x1, zf, sf, rf, qmax) << bits) |
                       ((uint32_t)affine_code(x2, zf, sf, rf, qmax) << (2 * bits)) |
                       ((uint32_t)affine_code(x3, zf, sf, rf, qmax) << (3 * bits));
    if (bits == 2)       // lanes 4j: channels 16j..16j+15
        wv = b | (__shfl_down_sync(0xFFFFFFFFu, b, 1) << 8) | (__shfl_down_sync(0xFFFFFFFFu, b, 2) << 16) |
             (__shfl_down_sync(0xFFFFFFFFu, b, 3) << 24);
    else                 // lanes 2j: channels 8j..8j+7, channel c at nibble c % 2 of byte c / 2
        wv = b | (__shfl_down_sync(0xFFFFFFFFu, b, 1) << 16);
}
template <int GV>
__device__ __forceinline__ void value_token_quant(const uint16_t *__restrict__ src, int lane, uint32_t &wv, uint16_t &s,
                                                  uint16_t &z, int bits = 2) {
    value_token_quant_x<GV>(*reinterpret_cast<const uint2 *>(src + 4 * lane), lane, wv, s, z, bits);
}

// Store of one token's packed codes by the lanes that hold a full word: token-major (the Kitty value pages,
// and KIVI values unless tiled), or into the KIVI value tiles of `codes` (token t of the row, lanes 4j
// holding channel quads 4j .. 4j + 3, one byte each).
__device__ __forceinline__ void value_token_store(uint8_t *__restrict__ tok, int lane, uint32_t wv, int bits) {
    if (bits == 2) {
        if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(tok)[lane >> 2] = wv;
    } else {
        if ((lane & 1) == 0) reinterpret_cast<uint32_t *>(tok)[lane >> 1] = wv;
    }
}
// Every lane calls it (a shuffle at 4 bits): there lanes 2j hold channels 8j .. 8j + 7 as nibbles, and lane
// 2j < 16 writes the bytes of channels 8j + k with 8j + k + 64 (from lane 2j + 16) in the high nibble.
__device__ __forceinline__ void value_token_store_kivi(uint8_t *__restrict__ codes, int64_t t, int lane, uint32_t wv,
                                                       int bits, bool tiles) {
    if (tiles && bits == 2) {
        if ((lane & 3) == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) codes[kivi_value_byte(t, lane + k)] = (uint8_t)(wv >> (8 * k));
        }
    } else if (tiles) {
        const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, wv, 16);
        if ((lane & 1) == 0 && lane < 16) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                codes[kivi_value_byte4(t, 4 * lane + k)] = (uint8_t)(((wv >> (4 * k)) & 15u) | (((hi >> (4 * k)) & 15u) << 4));
        }
    } else {
        value_token_store(codes + t * (KVQ_D * bits / 8), lane, wv, bits);
    }
}

// ---------------------------------------------------------------------------
// a2 / a6: per-token value quantization over groups of GV channels, in bulk.
// A warp takes four tokens at once: lane = 8 * token slot + channel block,
// the block's 16 channels (two 16-byte loads) in registers; group min / max
// by xor shuffles inside the GV/16 lanes of a group.  A lane's 16 codes are
// one word (2-bit: channel c at bits 2(c % 4) of byte c / 4) or two (4-bit:
// nibble c % 2 of byte c / 2) of the token's code row.  Output either KIVI
// (interleaved (s, z) per group) or a Kitty value page (separate s[G], z[G]
// after the codes).
// ---------------------------------------------------------------------------
template <int GV, bool KITTY, int BITS>
__global__ void __launch_bounds__(256, 3) quant_value_kernel(const uint16_t *__restrict__ v, int64_t n_tokens,
                                                          uint8_t *__restrict__ out, uint32_t *__restrict__ sz,
                                                          int page_tokens, int64_t page_bytes, bool tiles) {
    constexpr int LG = GV / 16, QMAX = (1 << BITS) - 1;   // lanes per group
    const int lane = threadIdx.x & 31, ts = lane >> 3, cb = lane & 7;
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    // the lane's 16 channels of token t, zeros past the end
    auto load = [&](int64_t t, uint4 &a, uint4 &b) {
        a = make_uint4(0u, 0u, 0u, 0u);
        b = a;
        if (t < n_tokens) {
            const uint4 *p = reinterpret_cast<const uint4 *>(v + t * KVQ_D + 16 * cb);
            a = __ldg(p);
            b = __ldg(p + 1);
        }
    };
    uint4 na, nb;                                   // the next pass's tokens, loaded while this pass codes
    load(4 * warp + ts, na, nb);
    for (int64_t t0 = 4 * warp; t0 < n_tokens; t0 += 4 * nwarps) {
        const int64_t t = t0 + ts;
        const bool live = t < n_tokens;
        const uint4 a = na, b = nb;
        load(t + 4 * nwarps, na, nb);
        const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        float x[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = h2f(lo16(h[i]));
            x[2 * i + 1] = h2f(hi16(h[i]));
        }
        float mn = x[0], mx = x[0];
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            mn = fminf(mn, x[i]);
            mx = fmaxf(mx, x[i]);
        }
#pragma unroll
        for (int o = 1; o < LG; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        }
        uint16_t s, z;
        affine_fit(mn, mx, QMAX, s, z);
        const float sf = h2f(s), zf = h2f(z), rf = sf != 0.0f ? __frcp_rn(sf) : 0.0f;
        uint32_t w[BITS / 2] = {};
        bool tie = false;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t code = (uint32_t)affine_code_fast(x[i], zf, rf, tie);
            if (BITS == 2) w[0] |= code << (2 * i);
            else w[i / 8] |= code << (4 * (i % 8));
        }
        if (tie) {                       // a near-tie: the lane's codes again with the quotient
#pragma unroll
            for (int i = 0; i < BITS / 2; ++i) w[i] = 0u;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t code = (uint32_t)affine_code(x[i], zf, sf, rf, QMAX);
                if (BITS == 2) w[0] |= code << (2 * i);
                else w[i / 8] |= code << (4 * (i % 8));
            }
        }
        // 4-bit tiles pair channel c with c + 64 in a byte: lane cb < 4 takes the codes of lane cb + 4
        uint32_t w64[2] = {0u, 0u};
        if constexpr (BITS == 4 && !KITTY) {
            if (tiles) {
                w64[0] = __shfl_down_sync(0xFFFFFFFFu, w[0], 4);
                w64[1] = __shfl_down_sync(0xFFFFFFFFu, w[1], 4);
            }
        }
        if (!live) continue;
        if (!KITTY) {
            if constexpr (BITS == 4) {
                if (tiles) {
                    // channels 16cb + k with 16cb + k + 64 in one byte of the 4-bit value tiles
                    if (cb < 4) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const uint32_t lo = (w[k / 8] >> (4 * (k % 8))) & 15u, hi = (w64[k / 8] >> (4 * (k % 8))) & 15u;
                            out[kivi_value_byte4(t, 16 * cb + k)] = (uint8_t)(lo | (hi << 4));
                        }
                    }
                } else {
                    reinterpret_cast<uint2 *>(out + t * (KVQ_D / 2))[cb] = make_uint2(w[0], w[1]);
                }
            } else if (tiles) {
                // channel quads 4cb .. 4cb + 3 of token t into the 32-token value tiles
#pragma unroll
                for (int k = 0; k < 4; ++k) out[kivi_value_byte(t, 4 * cb + k)] = (uint8_t)(w[0] >> (8 * k));
            } else {
                reinterpret_cast<uint32_t *>(out + t * (KVQ_D / 4))[cb] = w[0];
            }
            if (cb % LG == 0) sz[t * (KVQ_D / GV) + cb / LG] = (uint32_t)s | ((uint32_t)z << 16);
        } else {
            const int64_t p = t / page_tokens;
            const int tt = (int)(t % page_tokens);
            uint8_t *pg = out + p * page_bytes;
            reinterpret_cast<uint32_t *>(pg + (int64_t)tt * (KVQ_D / 4))[cb] = w[0];
            if (cb == 0) {
                uint16_t *ps = reinterpret_cast<uint16_t *>(pg + (int64_t)page_tokens * KVQ_D / 4);
                ps[tt] = s;
                ps[page_tokens + tt] = z;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// a5: Kitty key page.  One CTA of 128 threads per page (thread = channel);
// the page is staged in shared memory.  Score: Eq. 2 as an exact integer sum
// of |x| in units of 2^-24, or the sequential-fp32 population variance.
// Rank = number of channels with a larger score (ties: lower channel first);
// boosted iff rank < K; idx = boosted channels below this one.
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long abs_units(uint16_t h) {
    const int e = (h >> 10) & 0x1F, m = h & 0x3FF;
    return e == 0 ? (long long)m : ((long long)(1024 + m) << (e - 1));
}

// The codes of channel c of a key page into the shared copy of its planes:
// for tile j and token quad q, the low bits of tokens 32j + q + 8p (p = 0..3,
// bits 2p) at byte j*1024 + 64q + pos, and for a boosted channel of rank r
// the high bits at byte 4096 + j*8Kp + 4q + hpos.  With EXACT false the
// product form (affine_code_fast); the return value reports a near-tie.
template <bool EXACT>
__device__ __forceinline__ bool kitty_channel_codes(const uint16_t *xs, int c, float zf, float sf, float rf, int qmax,
                                                    uint8_t *cw, int pos, bool boosted, int hpos, int kp8, int j0,
                                                    int j1) {
    bool tie = false;
#pragma unroll 1
    for (int j = j0; j < j1; ++j)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t lo = 0u, hi = 0u;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float x = h2f(xs[(32 * j + q + 8 * p) * KVQ_D + c]);
                const uint32_t code = EXACT ? (uint32_t)affine_code(x, zf, sf, rf, qmax)
                                            : (uint32_t)affine_code_fast(x, zf, rf, tie);
                lo |= (code & 3u) << (2 * p);
                hi |= (code >> 2) << (2 * p);
            }
            cw[j * 1024 + q * 64 + pos] = (uint8_t)lo;
            if (boosted) cw[4096 + j * kp8 + q * 4 + hpos] = (uint8_t)hi;
        }
    return tie;
}

// Work area of a Kitty key page beside its fp16 copy, for a block of NT = 128 J threads (J threads per
// channel): the channels' rank keys and scores, the warps' boosted counts, the J threads' partial
// scores, extrema and ranks, and the planes' bytes (low 4096 B, high Kp * 32 B).
__host__ __device__ constexpr size_t kitty_key_work(int J) {
    return (size_t)KVQ_D * (8 + 4 + 4) + (size_t)J * KVQ_D * (8 + 4 + 4 + 4) + 4096 + 128 * 32;
}

// One Kitty key page (G = 128 tokens) by a block of NT threads from its fp16 copy xs [G][D] in shared
// memory, with `work` (kitty_key_work(NT / 128) bytes).  Thread (j, c) = (tid / 128, tid % 128) serves
// channel c and tokens [32 J' j, 32 J' (j + 1)), J' = 4 / J: its part of the exact score sum and the
// extrema (combined over the channel's J threads: integer sums and min / max do not depend on the order),
// its share of the rank comparisons, and the codes of its tiles.  The variance score (score_mode 1) is a
// sequential fp32 sum in token order, taken by the channel's thread j = 0.
template <int NT>
__device__ __forceinline__ void kitty_key_page_from_smem(const uint16_t *__restrict__ xs, int K, int score_mode,
                                                         uint8_t *__restrict__ pg, uint8_t *work) {
    constexpr int G = 128, J = NT / 128, TQ = G / J;
    unsigned long long *si = reinterpret_cast<unsigned long long *>(work);   // [D] rank keys (score mode 0)
    float *sf = reinterpret_cast<float *>(si + KVQ_D);                 // [D] variances (score mode 1)
    int *boost = reinterpret_cast<int *>(sf + KVQ_D);                   // [D] boosted channels per warp (4 used)
    long long *pa = reinterpret_cast<long long *>(boost + KVQ_D);      // [J][D] partial score sums
    float *pmn = reinterpret_cast<float *>(pa + J * KVQ_D);            // [J][D] partial minima
    float *pmx = pmn + J * KVQ_D;                                       // [J][D] partial maxima
    int *prk = reinterpret_cast<int *>(pmx + J * KVQ_D);                // [J][D] partial ranks
    uint8_t *cw = reinterpret_cast<uint8_t *>(prk + J * KVQ_D);        // the planes: low 4096 B, high Kp * 32 B
    const int Kp = kitty_high_rows(K);
    const int tid = threadIdx.x, c = tid & (KVQ_D - 1), j = tid / KVQ_D;
    for (int i = tid; i < Kp * 8; i += NT) reinterpret_cast<uint32_t *>(cw + 4096)[i] = 0u;   // rows past K stay 0
    long long a = 0;
    float mn = INFINITY, mx = -INFINITY, var = 0.f;
    if (score_mode == 0) {
#pragma unroll 4
        for (int t = j * TQ; t < (j + 1) * TQ; ++t) {
            const uint16_t h = xs[t * KVQ_D + c];
            const float x = h2f(h);
            a += abs_units(h);
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
    } else if (j == 0) {
        float s1 = 0.f, s2 = 0.f;
        for (int t = 0; t < G; ++t) {
            float x = h2f(xs[t * KVQ_D + c]);
            s1 = __fadd_rn(s1, x);
            s2 = __fadd_rn(s2, __fmul_rn(x, x));
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        float mean = __fdiv_rn(s1, (float)G);
        var = __fsub_rn(__fdiv_rn(s2, (float)G), __fmul_rn(mean, mean));
        sf[c] = var;
    }
    if (J > 1) {
        pa[j * KVQ_D + c] = a;
        pmn[j * KVQ_D + c] = mn;
        pmx[j * KVQ_D + c] = mx;
        __syncthreads();
        if (score_mode == 0) {
            a = 0;
            mn = INFINITY;
            mx = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < J; ++jj) {
                a += pa[jj * KVQ_D + c];
                mn = fminf(mn, pmn[jj * KVQ_D + c]);
                mx = fmaxf(mx, pmx[jj * KVQ_D + c]);
            }
        } else {
            mn = pmn[c];
            mx = pmx[c];
            var = sf[c];
        }
    }
    // mode 0: the score (below 2^47) and the channel as one key, (a << 7) | (127 - c): a larger key is a
    // larger score or, on a tie, a lower channel, so a channel's rank is the number of larger keys
    const unsigned long long key = ((unsigned long long)a << 7) | (unsigned long long)(127 - c);
    if (j == 0) si[c] = key;
    __syncthreads();
    int rank = 0;
    if (score_mode == 0) {
#pragma unroll 8
        for (int o = j * TQ; o < (j + 1) * TQ; ++o) rank += si[o] > key ? 1 : 0;
    } else {
        for (int o = j * TQ; o < (j + 1) * TQ; ++o) rank += (sf[o] > var || (sf[o] == var && o < c)) ? 1 : 0;
    }
    if (J > 1) {
        prk[j * KVQ_D + c] = rank;
        __syncthreads();
        rank = 0;
#pragma unroll
        for (int jj = 0; jj < J; ++jj) rank += prk[jj * KVQ_D + c];
    }
    const int boosted = rank < K;
    // r = boosted channels below c: a ballot within the warp (every warp holds 32 consecutive channels)
    // plus the counts of the channel warps below
    const unsigned bm = __ballot_sync(0xFFFFFFFFu, boosted);
    if (j == 0 && (c & 31) == 0) boost[c >> 5] = __popc(bm);
    __syncthreads();
    int r = __popc(bm & ((1u << (c & 31)) - 1u));
    for (int w = 0; w < (c >> 5); ++w) r += boost[w];
    const int qmax = boosted ? 15 : 3;
    uint16_t s, z;
    affine_fit(mn, mx, qmax, s, z);
    const float sv = h2f(s), zv = h2f(z), rv = sv != 0.0f ? __frcp_rn(sv) : 0.0f;
    // channel c = 16k + 2rr + e + 8h: byte (k/4)*512 + 16rr + (k%4)*4 + e + 2h of chunk row 4q + rr (the
    // KIVI key-tile order); boosted row r = 16kh + 4rb + b: byte 128kh + 32rb + b of a tile's high block
    const int k = c >> 4, cc = c & 15;
    const int pos = (k >> 2) * 512 + ((cc & 7) >> 1) * 16 + (k & 3) * 4 + (cc & 1) + 2 * (cc >> 3);
    const int hpos = (r >> 4) * 128 + ((r & 15) >> 2) * 32 + (r & 3);
    // the product form; tiles that met a near-tie are coded again with the quotient
    const int j0 = j * (4 / J), j1 = (j + 1) * (4 / J);
    if (kitty_channel_codes<false>(xs, c, zv, sv, rv, qmax, cw, pos, boosted, hpos, 8 * Kp, j0, j1))
        kitty_channel_codes<true>(xs, c, zv, sv, rv, qmax, cw, pos, boosted, hpos, 8 * Kp, j0, j1);
    if (j == 0) {
        uint8_t *idx = pg + KVQ_D * G / 4 + (int64_t)Kp * G / 4;
        uint16_t *ps = reinterpret_cast<uint16_t *>(idx + KVQ_D);
        idx[c] = boosted ? (uint8_t)r : (uint8_t)(K + 1);
        ps[c] = s;
        ps[KVQ_D + c] = z;
    }
    __syncthreads();
    // both planes (4096 + Kp * 32 bytes, a multiple of 16) with 16-byte stores
    const uint4 *c4 = reinterpret_cast<const uint4 *>(cw);
    uint4 *o4 = reinterpret_cast<uint4 *>(pg);
    for (int i = tid; i < (4096 + Kp * 32) / 16; i += NT) o4[i] = c4[i];
    __syncthreads();
}

// Shared memory of a block of NT threads quantizing key pages: the page's fp16 copy, then the work area.
__host__ __device__ constexpr size_t kitty_key_smem(int NT) { return (size_t)128 * KVQ_D * 2 + kitty_key_work(NT / 128); }
constexpr size_t KITTY_KEY_SMEM = kitty_key_smem(128);
constexpr int KITTY_KEY_BULK_NT = 256;   // the bulk and paged entry points: two threads per channel, 4 blocks per SM

// The same from global memory: the block copies the page into `smem` (G*D fp16, then the work area).
template <int NT>
__device__ __forceinline__ void kitty_key_page_quant(const uint16_t *__restrict__ src, int K, int score_mode,
                                                     uint8_t *__restrict__ pg, uint8_t *smem) {
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = threadIdx.x; i < 128 * KVQ_D / 8; i += NT) reinterpret_cast<uint4 *>(xs)[i] = s4[i];
    __syncthreads();
    kitty_key_page_from_smem<NT>(xs, K, score_mode, pg, smem + (size_t)128 * KVQ_D * 2);
}

__global__ void __launch_bounds__(KITTY_KEY_BULK_NT, 4) quant_key_kitty_kernel(const uint16_t *__restrict__ k,
                                                                               int64_t n_pages, int K, int score_mode,
                                                                               uint8_t *__restrict__ pages,
                                                                               int64_t page_bytes) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    for (int64_t p = blockIdx.x; p < n_pages; p += gridDim.x)
        kitty_key_page_quant<KITTY_KEY_BULK_NT>(k + p * (int64_t)128 * KVQ_D, K, score_mode, pages + p * page_bytes,
                                                smem_raw);
}

// ---------------------------------------------------------------------------
// a8: INT8 subtractive dither.  One CTA of 256 threads per block of T tokens;
// thread (warp w, lane l) owns channels 4l..4l+3 and tokens t = w (mod 8), so
// one Philox4x32-10 call yields the four dithers of its four channels.
// ---------------------------------------------------------------------------
// One INT8 block of T tokens by a 256-thread block: per-channel amax ->
// s = fp16_RN(amax / 126.5); code = clamp(rint(x / s + xi), -127, 127) with
// the Philox dither of (token t0 + t, channel, c2, c3) (WitCert section 6.1).
__device__ __forceinline__ void int8_block_quant(const uint16_t *__restrict__ xb, int T, uint32_t c2, uint32_t c3,
                                                 int32_t t0, uint32_t k0, uint32_t k1, int8_t *__restrict__ codes,
                                                 uint16_t *__restrict__ scale, float (*amax_part)[KVQ_D],
                                                 float *s_sh) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    for (int t = w; t < T; t += 8) {
        uint2 u = *reinterpret_cast<const uint2 *>(xb + (int64_t)t * KVQ_D + 4 * lane);
        a0 = fmaxf(a0, fabsf(h2f(lo16(u.x))));
        a1 = fmaxf(a1, fabsf(h2f(hi16(u.x))));
        a2 = fmaxf(a2, fabsf(h2f(lo16(u.y))));
        a3 = fmaxf(a3, fabsf(h2f(hi16(u.y))));
    }
    amax_part[w][4 * lane + 0] = a0;
    amax_part[w][4 * lane + 1] = a1;
    amax_part[w][4 * lane + 2] = a2;
    amax_part[w][4 * lane + 3] = a3;
    __syncthreads();
    if (threadIdx.x < KVQ_D) {
        float a = amax_part[0][threadIdx.x];
#pragma unroll
        for (int i = 1; i < 8; ++i) a = fmaxf(a, amax_part[i][threadIdx.x]);
        uint16_t s = f2h_rn(__fdiv_rn(a, 126.5f));
        scale[threadIdx.x] = s;
        s_sh[threadIdx.x] = h2f(s);
    }
    __syncthreads();
    const float s0 = s_sh[4 * lane], s1 = s_sh[4 * lane + 1], s2 = s_sh[4 * lane + 2], s3 = s_sh[4 * lane + 3];
    const float ri[4] = {s0 != 0.f ? __frcp_rn(s0) : 0.f, s1 != 0.f ? __frcp_rn(s1) : 0.f,
                         s2 != 0.f ? __frcp_rn(s2) : 0.f, s3 != 0.f ? __frcp_rn(s3) : 0.f};
    for (int t = w; t < T; t += 8) {
        uint4 r = philox4x32_10(make_uint4((uint32_t)(t0 + t), (uint32_t)lane, c2, c3), k0, k1);
        uint2 u = *reinterpret_cast<const uint2 *>(xb + (int64_t)t * KVQ_D + 4 * lane);
        float xs[4] = {h2f(lo16(u.x)), h2f(hi16(u.x)), h2f(lo16(u.y)), h2f(hi16(u.y))};
        float ss[4] = {s0, s1, s2, s3};
        uint32_t wr[4] = {r.x, r.y, r.z, r.w};
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int code = 0;
            if (ss[i] != 0.0f) code = dither_code(xs[i], ss[i], ri[i], dither_from_word(wr[i]));
            packed |= ((uint32_t)(code & 0xFF)) << (8 * i);
        }
        reinterpret_cast<uint32_t *>(codes + (int64_t)t * KVQ_D)[lane] = packed;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(256) quant_int8_kernel(const uint16_t *__restrict__ x, int64_t n_blocks, int T,
                                                         const int32_t *__restrict__ req,
                                                         const int32_t *__restrict__ head,
                                                         const int32_t *__restrict__ tok0, uint32_t ctr2_layer,
                                                         uint32_t k0, uint32_t k1, int8_t *__restrict__ codes,
                                                         uint16_t *__restrict__ scale) {
    __shared__ float amax_part[8][KVQ_D];
    __shared__ float s_sh[KVQ_D];
    for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
        const uint32_t c2 = ctr2_layer | ((uint32_t)head[b] & 0xFFFFu);
        int8_block_quant(x + b * (int64_t)T * KVQ_D, T, c2, (uint32_t)req[b], tok0[b], k0, k1,
                         codes + b * (int64_t)T * KVQ_D, scale + b * KVQ_D, amax_part, s_sh);
    }
}

__global__ void philox_kernel(const uint32_t *__restrict__ ctr, const uint32_t *__restrict__ key, int64_t n,
                              uint32_t *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        uint4 c = make_uint4(ctr[4 * i], ctr[4 * i + 1], ctr[4 * i + 2], ctr[4 * i + 3]);
        uint4 r = philox4x32_10(c, key[2 * i], key[2 * i + 1]);
        out[4 * i] = r.x; out[4 * i + 1] = r.y; out[4 * i + 2] = r.z; out[4 * i + 3] = r.w;
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int grid_cap(int64_t want, int per_sm) {
    int64_t cap = (int64_t)num_sms() * per_sm;
    return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

cudaError_t launch_quant_key_kivi(const kvq_config *cfg, const void *k, int64_t n_groups, void *codes, void *sz,
                                  cudaStream_t st) {
    if (n_groups == 0) return cudaSuccess;
    const uint16_t *kp = static_cast<const uint16_t *>(k);
    uint8_t *cp = static_cast<uint8_t *>(codes);
    uint16_t *zp = static_cast<uint16_t *>(sz);
    // one CTA per group; grids above 2^31-1 groups are split into launches
    for (int64_t g0 = 0; g0 < n_groups; g0 += 0x7FFFFFFF) {
        int64_t n = n_groups - g0 < 0x7FFFFFFF ? n_groups - g0 : 0x7FFFFFFF;
        const int G = cfg->group_k;
        const uint16_t *ks = kp + g0 * (int64_t)G * KVQ_D;
        uint8_t *cs = cp + g0 * (int64_t)G * KVQ_D * cfg->bits_k / 8;
        uint16_t *zs = zp + g0 * 2 * KVQ_D;
        const int bits = cfg->bits_k;
        const unsigned grid = (unsigned)grid_cap(n, G == 32 ? 12 : G == 64 ? 6 : 4);   // resident blocks per SM
        const bool b4 = bits == 4;
        if (G == 32) {
            if (b4) quant_key_kivi_kernel<1, 4><<<grid, 128, 0, st>>>(ks, n, cs, zs);
            else quant_key_kivi_kernel<1, 2><<<grid, 128, 0, st>>>(ks, n, cs, zs);
        } else if (G == 64) {
            if (b4) quant_key_kivi_kernel<2, 4><<<grid, 128, 0, st>>>(ks, n, cs, zs);
            else quant_key_kivi_kernel<2, 2><<<grid, 128, 0, st>>>(ks, n, cs, zs);
        } else {
            if (b4) quant_key_kivi_kernel<4, 4><<<grid, 128, 0, st>>>(ks, n, cs, zs);
            else quant_key_kivi_kernel<4, 2><<<grid, 128, 0, st>>>(ks, n, cs, zs);
        }
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_value_kivi(const kvq_config *cfg, const void *v, int64_t n_tokens, void *codes, void *sz,
                                    cudaStream_t st) {
    if (n_tokens == 0) return cudaSuccess;
    const int grid = grid_cap((n_tokens + 31) / 32, 3);           // 32 tokens per 8-warp block pass; 3 resident
    const uint16_t *vp = static_cast<const uint16_t *>(v);
    uint8_t *cp = static_cast<uint8_t *>(codes);
    uint32_t *zp = static_cast<uint32_t *>(sz);
    const bool tiles = kivi_value_tiles(cfg);
#define KVQ_QV(GV, B) quant_value_kernel<GV, false, B><<<grid, 256, 0, st>>>(vp, n_tokens, cp, zp, 0, 0, tiles)
    const bool b4 = cfg->bits_v == 4;
    switch (cfg->group_v) {
        case 32: if (b4) KVQ_QV(32, 4); else KVQ_QV(32, 2); break;
        case 64: if (b4) KVQ_QV(64, 4); else KVQ_QV(64, 2); break;
        default: if (b4) KVQ_QV(128, 4); else KVQ_QV(128, 2); break;
    }
#undef KVQ_QV
    return cudaGetLastError();
}

cudaError_t launch_quant_value_kitty(const kvq_config *cfg, const void *v, int64_t n_pages, void *pages,
                                     cudaStream_t st) {
    if (n_pages == 0) return cudaSuccess;
    const int G = cfg->group_k;
    const int64_t n_tokens = n_pages * G;
    const int grid = grid_cap((n_tokens + 31) / 32, 3);
    const int64_t pb = (int64_t)G * KVQ_D / 4 + 4LL * G;
    quant_value_kernel<128, true, 2><<<grid, 256, 0, st>>>(static_cast<const uint16_t *>(v), n_tokens,
                                                           static_cast<uint8_t *>(pages), nullptr, G, pb, false);
    return cudaGetLastError();
}

cudaError_t launch_quant_key_kitty(const kvq_config *cfg, const void *k, int64_t n_pages, int score_mode,
                                   void *pages, cudaStream_t st) {
    if (n_pages == 0) return cudaSuccess;
    const int K = cfg->boost_k;
    const int64_t pb = kitty_key_page_bytes(K);
    const size_t smem = kitty_key_smem(KITTY_KEY_BULK_NT);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(quant_key_kitty_kernel, smem, attr_done)) return e;
    const int grid = grid_cap(n_pages, 4);
    quant_key_kitty_kernel<<<grid, KITTY_KEY_BULK_NT, smem, st>>>(static_cast<const uint16_t *>(k), n_pages, K,
                                                                  score_mode, static_cast<uint8_t *>(pages), pb);
    return cudaGetLastError();
}

cudaError_t launch_quant_int8(const kvq_config *cfg, const void *x, int64_t n_blocks, const int32_t *req,
                              const int32_t *head, const int32_t *tok0, int layer, int kv_sel, uint64_t seed,
                              void *codes, void *scale, cudaStream_t st) {
    if (n_blocks == 0) return cudaSuccess;
    const uint32_t c2 = ((uint32_t)layer << 17) | ((uint32_t)(kv_sel & 1) << 16);
    const int grid = grid_cap(n_blocks, 8);
    quant_int8_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t *>(x), n_blocks, cfg->int8_block, req, head,
                                            tok0, c2, (uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32),
                                            static_cast<int8_t *>(codes), static_cast<uint16_t *>(scale));
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Streaming append (KIVI): one CTA of 128 threads per (batch row, kv head).
// With L = seq_len[b] tokens cached, it first finishes the quantization that
// follows the attention of the step with L tokens (the order is insert ->
// attend -> quantize), then inserts token L:
//   * keys: when L is a positive multiple of R the full key residual
//     [L-R, L) (ring slots 0..R-1) becomes R/G quantized groups;
//   * values: when L >= R, token L-R leaves the fp16 window and is quantized;
//   * the new k, v are written to ring slot L % R.
// The quantizers are the ones of kv_quant_key / kv_quant_value, so appending
// token by token gives the bytes of a cache filled at once.  A second kernel
// bumps seq_len once every head has read it.
// ---------------------------------------------------------------------------
struct AppendParams {
    const int32_t *seq_len;
    const uint16_t *k_new, *v_new;
    uint8_t *k_codes, *v_codes;
    uint16_t *k_sz;
    uint32_t *v_sz;
    uint16_t *k_res, *v_res;
    unsigned *err;
    int Hkv, R, G, ngv, max_seq_len, bits_k, bits_v;
    int vtiles;                  // values stored in value tiles (kivi_value_tiles)
    int64_t cap, kgrp_cap;
};

template <int NT, int GV>
__global__ void __launch_bounds__(128) append_kivi_kernel(AppendParams P) {
    const int64_t bk = blockIdx.x;
    const int b = (int)(bk / P.Hkv);
    const int L = P.seq_len[b];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (L < 0 || L >= P.max_seq_len) {
        if (threadIdx.x == 0) atomicOr(P.err, KVQ_DEVICE_ERR_CAPACITY);
        return;
    }
    constexpr int G = 32 * NT;
    const uint16_t *kres = P.k_res + bk * P.R * KVQ_D;
    const uint16_t *vres = P.v_res + bk * P.R * KVQ_D;
    if (L > 0 && L % P.R == 0) {
        for (int g = 0; g < P.R / G; ++g) {
            const int64_t gi = bk * P.kgrp_cap + (L - P.R) / G + g;
            key_group_quant<NT>(kres + (int64_t)g * G * KVQ_D, P.k_codes + gi * (G * KVQ_D * P.bits_k / 8),
                                P.k_sz + gi * 2 * KVQ_D, P.bits_k);
        }
    }
    if (L >= P.R && warp == 0) {
        const int64_t t = L - P.R;
        uint32_t wv;
        uint16_t s, z;
        value_token_quant<GV>(vres + (t % P.R) * KVQ_D, lane, wv, s, z, P.bits_v);
        value_token_store_kivi(P.v_codes + bk * P.cap * (KVQ_D * P.bits_v / 8), t, lane, wv, P.bits_v, P.vtiles);
        if ((lane % (GV / 4)) == 0)
            P.v_sz[(bk * P.cap + t) * P.ngv + lane / (GV / 4)] = (uint32_t)s | ((uint32_t)z << 16);
    }
    __syncthreads();   // every read of the ring slot about to be overwritten is done
    const int64_t slot = L % P.R;
    if (threadIdx.x < 16) {
        reinterpret_cast<uint4 *>(P.k_res + (bk * P.R + slot) * KVQ_D)[threadIdx.x] =
            reinterpret_cast<const uint4 *>(P.k_new + bk * KVQ_D)[threadIdx.x];
    } else if (threadIdx.x < 32) {
        reinterpret_cast<uint4 *>(P.v_res + (bk * P.R + slot) * KVQ_D)[threadIdx.x - 16] =
            reinterpret_cast<const uint4 *>(P.v_new + bk * KVQ_D)[threadIdx.x - 16];
    }
}

__global__ void append_bump_kernel(int32_t *seq_len, int B, int max_seq_len) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B && seq_len[b] >= 0 && seq_len[b] < max_seq_len) seq_len[b] += 1;
}

cudaError_t launch_append_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *k_new, const void *v_new,
                               cudaStream_t st) {
    AppendParams P;
    P.seq_len = c->seq_len;
    P.k_new = static_cast<const uint16_t *>(k_new);
    P.v_new = static_cast<const uint16_t *>(v_new);
    P.k_codes = static_cast<uint8_t *>(const_cast<void *>(c->k_codes));
    P.v_codes = static_cast<uint8_t *>(const_cast<void *>(c->v_codes));
    P.k_sz = static_cast<uint16_t *>(const_cast<void *>(c->k_sz));
    P.v_sz = static_cast<uint32_t *>(const_cast<void *>(c->v_sz));
    P.k_res = static_cast<uint16_t *>(const_cast<void *>(c->k_res));
    P.v_res = static_cast<uint16_t *>(const_cast<void *>(c->v_res));
    P.err = device_error_ptr();
    if (!P.err) return cudaErrorInvalidDevicePointer;
    P.Hkv = cfg->n_kv_heads;
    P.R = cfg->residual;
    P.G = cfg->group_k;
    P.ngv = KVQ_D / cfg->group_v;
    P.bits_k = cfg->bits_k;
    P.bits_v = cfg->bits_v;
    P.vtiles = kivi_value_tiles(cfg);
    P.max_seq_len = c->max_seq_len;
    P.cap = ((int64_t)c->max_seq_len + 127) / 128 * 128;
    P.kgrp_cap = P.cap / cfg->group_k;
    const unsigned grid = (unsigned)((int64_t)c->batch * cfg->n_kv_heads);
#define KVQ_APPEND(NT, GV) append_kivi_kernel<NT, GV><<<grid, 128, 0, st>>>(P)
    const int G = cfg->group_k, GV = cfg->group_v;
    if (G == 32) { if (GV == 32) KVQ_APPEND(1, 32); else if (GV == 64) KVQ_APPEND(1, 64); else KVQ_APPEND(1, 128); }
    else if (G == 64) { if (GV == 32) KVQ_APPEND(2, 32); else if (GV == 64) KVQ_APPEND(2, 64); else KVQ_APPEND(2, 128); }
    else { if (GV == 32) KVQ_APPEND(4, 32); else if (GV == 64) KVQ_APPEND(4, 64); else KVQ_APPEND(4, 128); }
#undef KVQ_APPEND
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    append_bump_kernel<<<(c->batch + 127) / 128, 128, 0, st>>>(const_cast<int32_t *>(c->seq_len), c->batch,
                                                                c->max_seq_len);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Paged KIVI: a page record holds 128 tokens of one kv head in decode-stage
// order (key codes, key (s, z) 2048 B, value codes, value (s, z) 2048 B).
// The write side quantizes with the same device functions as the dense
// cache and only addresses through the page table.
// ---------------------------------------------------------------------------
struct PagedDst {
    const int32_t *page_table;
    uint8_t *pages;
    int pt_stride, n_pages, Hkv;
    int64_t rec_bytes;
    int kc_bytes, vc_bytes;
    int vtiles;                  // values stored in value tiles (kivi_value_tiles)
    unsigned *err;
};

// Record of logical page lp of row b, kv head h; null (KVQ_DEVICE_ERR_POOL
// recorded) when the table entry is outside the pool.
__device__ __forceinline__ uint8_t *paged_record(const PagedDst &D, int b, int lp, int h) {
    const int pg = D.page_table[(int64_t)b * D.pt_stride + lp];
    if (pg < 0 || pg >= D.n_pages) {
        if (threadIdx.x == 0) atomicOr(D.err, KVQ_DEVICE_ERR_POOL);
        return nullptr;
    }
    return D.pages + ((int64_t)pg * D.Hkv + h) * D.rec_bytes;
}

template <int NT>
__global__ void __launch_bounds__(128) quant_key_paged_kernel(const uint16_t *__restrict__ k, int64_t n_groups,
                                                              int group0, int row, int kvh, PagedDst D, int bits) {
    const int64_t g = blockIdx.x;
    if (g >= n_groups) return;
    constexpr int G = 32 * NT;
    const int gl = group0 + (int)g;
    uint8_t *rec = paged_record(D, row, gl * G / 128, kvh);
    if (!rec) return;
    const int gp = gl % (128 / G);
    key_group_quant<NT>(k + g * (int64_t)G * KVQ_D, rec + gp * (G * KVQ_D * bits / 8),
                        reinterpret_cast<uint16_t *>(rec + D.kc_bytes + gp * 512), bits);
}

// value token tg of the row (fp16 src) into its page record, by one warp
template <int GV>
__device__ __forceinline__ void value_token_paged(const uint16_t *__restrict__ src, uint8_t *rec, int tg,
                                                  const PagedDst &D, int ngv, int lane, int bits) {
    constexpr int LG = GV / 4;
    uint32_t wv;
    uint16_t s, z;
    value_token_quant<GV>(src, lane, wv, s, z, bits);
    const int tp = tg & 127;
    value_token_store_kivi(rec + D.kc_bytes + 2048, tp, lane, wv, bits, D.vtiles);
    if ((lane % LG) == 0)
        reinterpret_cast<uint32_t *>(rec + D.kc_bytes + 2048 + D.vc_bytes)[tp * ngv + lane / LG] =
            (uint32_t)s | ((uint32_t)z << 16);
}

template <int GV>
__global__ void __launch_bounds__(256) quant_value_paged_kernel(const uint16_t *__restrict__ v, int64_t n_tokens,
                                                                int tok0, int row, int kvh, PagedDst D, int ngv,
                                                                int bits) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tokens; t += nwarps) {
        const int tg = tok0 + (int)t;
        const int pg = D.page_table[(int64_t)row * D.pt_stride + (tg >> 7)];
        if (pg < 0 || pg >= D.n_pages) {
            if (lane == 0) atomicOr(D.err, KVQ_DEVICE_ERR_POOL);
            continue;
        }
        value_token_paged<GV>(v + t * KVQ_D, D.pages + ((int64_t)pg * D.Hkv + kvh) * D.rec_bytes, tg, D, ngv, lane,
                              bits);
    }
}

static PagedDst paged_dst(const kvq_config *cfg, const kvq_kivi_paged_cache *c) {
    PagedDst D;
    D.page_table = c->page_table;
    D.pages = static_cast<uint8_t *>(const_cast<void *>(c->pages));
    D.pt_stride = (int)(((int64_t)c->max_seq_len + 127) / 128);
    D.n_pages = c->n_pages;
    D.Hkv = cfg->n_kv_heads;
    D.rec_bytes = kivi_page_bytes(cfg->bits_k, cfg->bits_v);
    D.kc_bytes = 16 * KVQ_D * cfg->bits_k;
    D.vc_bytes = 16 * KVQ_D * cfg->bits_v;
    D.vtiles = kivi_value_tiles(cfg);
    D.err = device_error_ptr();
    return D;
}

cudaError_t launch_quant_key_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *k, int64_t n,
                                   int group0, int row, int kvh, cudaStream_t st) {
    const PagedDst D = paged_dst(cfg, c);
    if (!D.err) return cudaErrorInvalidDevicePointer;
    const uint16_t *kp = static_cast<const uint16_t *>(k);
    const int G = cfg->group_k, bits = cfg->bits_k;
    if (G == 32) quant_key_paged_kernel<1><<<(unsigned)n, 128, 0, st>>>(kp, n, group0, row, kvh, D, bits);
    else if (G == 64) quant_key_paged_kernel<2><<<(unsigned)n, 128, 0, st>>>(kp, n, group0, row, kvh, D, bits);
    else quant_key_paged_kernel<4><<<(unsigned)n, 128, 0, st>>>(kp, n, group0, row, kvh, D, bits);
    return cudaGetLastError();
}

cudaError_t launch_quant_value_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const void *v, int64_t n,
                                     int tok0, int row, int kvh, cudaStream_t st) {
    const PagedDst D = paged_dst(cfg, c);
    if (!D.err) return cudaErrorInvalidDevicePointer;
    const uint16_t *vp = static_cast<const uint16_t *>(v);
    int64_t grid = (n + 7) / 8;
    if (grid > (int64_t)num_sms() * 16) grid = (int64_t)num_sms() * 16;
    const int ngv = KVQ_D / cfg->group_v, bits = cfg->bits_v;
    switch (cfg->group_v) {
        case 32: quant_value_paged_kernel<32><<<(unsigned)grid, 256, 0, st>>>(vp, n, tok0, row, kvh, D, ngv, bits); break;
        case 64: quant_value_paged_kernel<64><<<(unsigned)grid, 256, 0, st>>>(vp, n, tok0, row, kvh, D, ngv, bits); break;
        default: quant_value_paged_kernel<128><<<(unsigned)grid, 256, 0, st>>>(vp, n, tok0, row, kvh, D, ngv, bits); break;
    }
    return cudaGetLastError();
}

// Streaming append into a paged cache: as append_kivi_kernel, with the key
// groups and the value token written into the row's page records.  A row
// whose new page could not be allocated (table entry -1) is left unchanged.
template <int NT, int GV>
__global__ void __launch_bounds__(128) append_kivi_paged_kernel(AppendParams P, PagedDst D) {
    const int64_t bk = blockIdx.x;
    const int b = (int)(bk / P.Hkv), h = (int)(bk % P.Hkv);
    const int L = P.seq_len[b];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (L < 0 || L >= P.max_seq_len) return;                // the allocator recorded the capacity error
    if ((L & 127) == 0 && D.page_table[(int64_t)b * D.pt_stride + (L >> 7)] < 0) return;
    constexpr int G = 32 * NT;
    const uint16_t *kres = P.k_res + bk * P.R * KVQ_D;
    const uint16_t *vres = P.v_res + bk * P.R * KVQ_D;
    if (L > 0 && L % P.R == 0) {
        for (int g = 0; g < P.R / G; ++g) {
            const int gl = (L - P.R) / G + g;
            uint8_t *rec = paged_record(D, b, gl * G / 128, h);
            if (!rec) continue;
            const int gp = gl % (128 / G);
            key_group_quant<NT>(kres + (int64_t)g * G * KVQ_D, rec + gp * (G * KVQ_D * P.bits_k / 8),
                                reinterpret_cast<uint16_t *>(rec + D.kc_bytes + gp * 512), P.bits_k);
        }
    }
    if (L >= P.R && warp == 0) {
        const int t = L - P.R;
        const int pg = D.page_table[(int64_t)b * D.pt_stride + (t >> 7)];
        if (pg >= 0 && pg < D.n_pages)
            value_token_paged<GV>(vres + (int64_t)(t % P.R) * KVQ_D, D.pages + ((int64_t)pg * D.Hkv + h) * D.rec_bytes,
                                  t, D, P.ngv, lane, P.bits_v);
        else if (lane == 0)
            atomicOr(D.err, KVQ_DEVICE_ERR_POOL);
    }
    __syncthreads();   // every read of the ring slot about to be overwritten is done
    const int64_t slot = L % P.R;
    if (threadIdx.x < 16) {
        reinterpret_cast<uint4 *>(P.k_res + (bk * P.R + slot) * KVQ_D)[threadIdx.x] =
            reinterpret_cast<const uint4 *>(P.k_new + bk * KVQ_D)[threadIdx.x];
    } else if (threadIdx.x < 32) {
        reinterpret_cast<uint4 *>(P.v_res + (bk * P.R + slot) * KVQ_D)[threadIdx.x - 16] =
            reinterpret_cast<const uint4 *>(P.v_new + bk * KVQ_D)[threadIdx.x - 16];
    }
}

// seq_len += 1 for every row that could append: not full, and not waiting
// for a page the allocator could not give (pages start after `base` tokens)
__global__ void append_bump_paged_kernel(int32_t *seq_len, const int32_t *table, int stride, int base, int B,
                                         int max_seq_len) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int L = seq_len[b];
    if (L < 0 || L >= max_seq_len) return;
    if (L >= base && ((L - base) & 127) == 0 && table[(int64_t)b * stride + ((L - base) >> 7)] < 0) return;
    seq_len[b] = L + 1;
}

cudaError_t launch_append_kivi_paged(const kvq_config *cfg, const kvq_kivi_paged_cache *c, const kvq_slot_pool *pool,
                                     const void *k_new, const void *v_new, cudaStream_t st) {
    const PagedDst D = paged_dst(cfg, c);
    if (!D.err) return cudaErrorInvalidDevicePointer;
    int32_t *seq_len = const_cast<int32_t *>(c->seq_len);
    cudaError_t e = launch_alloc_ids(seq_len, const_cast<int32_t *>(c->page_table), c->batch, c->max_seq_len, 128,
                                     D.pt_stride, 0, pool, st);
    if (e != cudaSuccess) return e;
    AppendParams P;
    P.seq_len = c->seq_len;
    P.k_new = static_cast<const uint16_t *>(k_new);
    P.v_new = static_cast<const uint16_t *>(v_new);
    P.k_codes = nullptr;
    P.v_codes = nullptr;
    P.k_sz = nullptr;
    P.v_sz = nullptr;
    P.k_res = static_cast<uint16_t *>(const_cast<void *>(c->k_res));
    P.v_res = static_cast<uint16_t *>(const_cast<void *>(c->v_res));
    P.err = D.err;
    P.Hkv = cfg->n_kv_heads;
    P.R = cfg->residual;
    P.G = cfg->group_k;
    P.ngv = KVQ_D / cfg->group_v;
    P.bits_k = cfg->bits_k;
    P.bits_v = cfg->bits_v;
    P.vtiles = kivi_value_tiles(cfg);
    P.max_seq_len = c->max_seq_len;
    P.cap = 0;
    P.kgrp_cap = 0;
    const int64_t grid = (int64_t)c->batch * cfg->n_kv_heads;
#define KVQ_APPEND_PAGED(NT, GV) append_kivi_paged_kernel<NT, GV><<<(unsigned)grid, 128, 0, st>>>(P, D)
    const int G = cfg->group_k, GV = cfg->group_v;
    if (G == 32) { if (GV == 32) KVQ_APPEND_PAGED(1, 32); else if (GV == 64) KVQ_APPEND_PAGED(1, 64); else KVQ_APPEND_PAGED(1, 128); }
    else if (G == 64) { if (GV == 32) KVQ_APPEND_PAGED(2, 32); else if (GV == 64) KVQ_APPEND_PAGED(2, 64); else KVQ_APPEND_PAGED(2, 128); }
    else { if (GV == 32) KVQ_APPEND_PAGED(4, 32); else if (GV == 64) KVQ_APPEND_PAGED(4, 64); else KVQ_APPEND_PAGED(4, 128); }
#undef KVQ_APPEND_PAGED
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    append_bump_paged_kernel<<<(c->batch + 127) / 128, 128, 0, st>>>(seq_len, c->page_table, D.pt_stride, 0,
                                                                      c->batch, c->max_seq_len);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Streaming append (INT8): one CTA of 256 threads per (batch row, kv head).
// With L = seq_len[b] cached: when L is a positive multiple of T the fp16
// tail [L-T, L) (ring slots 0..T-1) becomes the INT8 block (L-T)/T of K and V
// (the write kernel's quantizer and dither streams); then token L goes to tail
// slot L % T.  seq_len is bumped by a second kernel.
// ---------------------------------------------------------------------------
struct AppendInt8Params {
    const int32_t *seq_len, *req_id;
    const uint16_t *k_new, *v_new;
    int8_t *k_codes, *v_codes;
    uint16_t *k_scale, *v_scale, *k_tail, *v_tail;
    unsigned *err;
    int Hkv, T, max_seq_len, blk_cap;
    uint32_t ctr2_layer, k0, k1;
};

__global__ void __launch_bounds__(256) append_int8_kernel(AppendInt8Params P) {
    __shared__ float amax_part[8][KVQ_D];
    __shared__ float s_sh[KVQ_D];
    const int64_t bk = blockIdx.x;
    const int b = (int)(bk / P.Hkv), h = (int)(bk % P.Hkv);
    const int L = P.seq_len[b];
    if (L < 0 || L >= P.max_seq_len) {
        if (threadIdx.x == 0) atomicOr(P.err, KVQ_DEVICE_ERR_CAPACITY);
        return;
    }
    const int T = P.T;
    if (L > 0 && L % T == 0) {
        const int blk = (L - T) / T;
        const uint32_t c2 = P.ctr2_layer | ((uint32_t)h & 0xFFFFu);
        const uint32_t c3 = (uint32_t)P.req_id[b];
        int8_block_quant(P.k_tail + bk * T * KVQ_D, T, c2, c3, L - T, P.k0, P.k1,
                         P.k_codes + (bk * P.max_seq_len + (L - T)) * KVQ_D, P.k_scale + (bk * P.blk_cap + blk) * KVQ_D,
                         amax_part, s_sh);
        int8_block_quant(P.v_tail + bk * T * KVQ_D, T, c2 | 0x10000u, c3, L - T, P.k0, P.k1,
                         P.v_codes + (bk * P.max_seq_len + (L - T)) * KVQ_D, P.v_scale + (bk * P.blk_cap + blk) * KVQ_D,
                         amax_part, s_sh);
    }
    __syncthreads();
    const int64_t slot = L % T;
    if (threadIdx.x < 16) {
        reinterpret_cast<uint4 *>(P.k_tail + (bk * T + slot) * KVQ_D)[threadIdx.x] =
            reinterpret_cast<const uint4 *>(P.k_new + bk * KVQ_D)[threadIdx.x];
    } else if (threadIdx.x < 32) {
        reinterpret_cast<uint4 *>(P.v_tail + (bk * T + slot) * KVQ_D)[threadIdx.x - 16] =
            reinterpret_cast<const uint4 *>(P.v_new + bk * KVQ_D)[threadIdx.x - 16];
    }
}

cudaError_t launch_append_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *k_new, const void *v_new,
                               cudaStream_t st) {
    AppendInt8Params P;
    P.seq_len = c->seq_len;
    P.req_id = c->req_id;
    P.k_new = static_cast<const uint16_t *>(k_new);
    P.v_new = static_cast<const uint16_t *>(v_new);
    P.k_codes = static_cast<int8_t *>(const_cast<void *>(c->k_codes));
    P.v_codes = static_cast<int8_t *>(const_cast<void *>(c->v_codes));
    P.k_scale = static_cast<uint16_t *>(const_cast<void *>(c->k_scale));
    P.v_scale = static_cast<uint16_t *>(const_cast<void *>(c->v_scale));
    P.k_tail = static_cast<uint16_t *>(const_cast<void *>(c->k_tail));
    P.v_tail = static_cast<uint16_t *>(const_cast<void *>(c->v_tail));
    P.err = device_error_ptr();
    if (!P.err) return cudaErrorInvalidDevicePointer;
    P.Hkv = cfg->n_kv_heads;
    P.T = cfg->int8_block;
    P.max_seq_len = c->max_seq_len;
    P.blk_cap = (c->max_seq_len + P.T - 1) / P.T;
    if (P.blk_cap < 1) P.blk_cap = 1;
    P.ctr2_layer = (uint32_t)c->layer << 17;
    P.k0 = (uint32_t)(c->seed & 0xFFFFFFFFu);
    P.k1 = (uint32_t)(c->seed >> 32);
    append_int8_kernel<<<(unsigned)((int64_t)c->batch * cfg->n_kv_heads), 256, 0, st>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    append_bump_kernel<<<(c->batch + 127) / 128, 128, 0, st>>>(const_cast<int32_t *>(c->seq_len), c->batch,
                                                                c->max_seq_len);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Paged Kitty bulk writes: whole key / value pages of one kv head into the
// pool pages of a request's page table (the same page quantizers).
// ---------------------------------------------------------------------------
struct KittyPagedDst {
    const int32_t *page_table;
    uint8_t *pool;
    int page_cap, n_pages, Hkv, row, kvh, page0;
    int64_t rec_bytes;
    unsigned *err;
};

__device__ __forceinline__ uint8_t *kitty_paged_record(const KittyPagedDst &D, int p) {
    const int pg = D.page_table[(int64_t)D.row * D.page_cap + D.page0 + p];
    if (pg < 0 || pg >= D.n_pages) return nullptr;
    return D.pool + ((int64_t)pg * D.Hkv + D.kvh) * D.rec_bytes;
}

__global__ void __launch_bounds__(KITTY_KEY_BULK_NT, 4) quant_key_kitty_paged_kernel(const uint16_t *__restrict__ k,
                                                                                     int64_t n_pages, int K,
                                                                                     int score_mode, KittyPagedDst D) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    for (int64_t p = blockIdx.x; p < n_pages; p += gridDim.x) {
        uint8_t *rec = kitty_paged_record(D, (int)p);
        if (!rec) {
            if (threadIdx.x == 0) atomicOr(D.err, KVQ_DEVICE_ERR_POOL);
            continue;
        }
        kitty_key_page_quant<KITTY_KEY_BULK_NT>(k + p * (int64_t)128 * KVQ_D, K, score_mode, rec, smem_raw);
    }
}

__global__ void __launch_bounds__(256) quant_value_kitty_paged_kernel(const uint16_t *__restrict__ v, int64_t n_tokens,
                                                                      KittyPagedDst D) {
    constexpr int G = 128;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < n_tokens; t += nwarps) {
        uint8_t *pg = kitty_paged_record(D, (int)(t / G));
        if (!pg) {
            if (lane == 0) atomicOr(D.err, KVQ_DEVICE_ERR_POOL);
            continue;
        }
        const int tt = (int)(t % G);
        uint32_t wv;
        uint16_t sv, zv;
        value_token_quant<128>(v + t * KVQ_D, lane, wv, sv, zv);
        if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(pg + (int64_t)tt * (KVQ_D / 4))[lane >> 2] = wv;
        if (lane == 0) {
            uint16_t *ps = reinterpret_cast<uint16_t *>(pg + (int64_t)G * KVQ_D / 4);
            ps[tt] = sv;
            ps[G + tt] = zv;
        }
    }
}

static KittyPagedDst kitty_paged_dst(const kvq_config *cfg, const kvq_kitty_cache *c, const void *pool, int64_t rec,
                                     int page0, int row, int kvh) {
    KittyPagedDst D;
    D.page_table = c->page_table;
    D.pool = static_cast<uint8_t *>(const_cast<void *>(pool));
    D.page_cap = (int)((c->max_seq_len - cfg->sink > 0 ? c->max_seq_len - cfg->sink : 0) + 127) / 128;
    if (D.page_cap < 1) D.page_cap = 1;
    D.n_pages = c->n_pages;
    D.Hkv = cfg->n_kv_heads;
    D.row = row;
    D.kvh = kvh;
    D.page0 = page0;
    D.rec_bytes = rec;
    D.err = device_error_ptr();
    return D;
}

cudaError_t launch_quant_key_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k, int64_t n,
                                         int page0, int row, int kvh, int score_mode, cudaStream_t st) {
    const int64_t kpb = kitty_key_page_bytes(cfg->boost_k);
    const KittyPagedDst D = kitty_paged_dst(cfg, c, c->k_pages, kpb, page0, row, kvh);
    if (!D.err) return cudaErrorInvalidDevicePointer;
    static std::atomic<uint64_t> attr_done{0};
    const size_t smem = kitty_key_smem(KITTY_KEY_BULK_NT);
    if (cudaError_t e = smem_opt_in(quant_key_kitty_paged_kernel, smem, attr_done)) return e;
    const int grid = grid_cap(n, 4);
    quant_key_kitty_paged_kernel<<<grid, KITTY_KEY_BULK_NT, smem, st>>>(static_cast<const uint16_t *>(k), n,
                                                                        cfg->boost_k, score_mode, D);
    return cudaGetLastError();
}

cudaError_t launch_quant_value_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const void *v, int64_t n,
                                           int page0, int row, int kvh, cudaStream_t st) {
    const int64_t vpb = 128LL * KVQ_D / 4 + 4LL * 128;
    const KittyPagedDst D = kitty_paged_dst(cfg, c, c->v_pages, vpb, page0, row, kvh);
    if (!D.err) return cudaErrorInvalidDevicePointer;
    const int64_t n_tokens = n * 128;
    const int grid = grid_cap((n_tokens + 7) / 8, 16);
    quant_value_kitty_paged_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t *>(v), n_tokens, D);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Streaming append (Kitty): one CTA of 128 threads per (batch row, kv head).
// With L = seq_len[b] cached it completes the quantization that follows the
// attention of the step with L tokens, then inserts token L (Kitty, "Stage 1:
// Inserting New KV Vectors" and "Stage 3" of the pipeline):
//   * keys: when (L - S) is a positive multiple of G the full key Q-buffer
//     becomes key page (L - S)/G - 1;
//   * values: when E = L - S - R is a positive multiple of G the full value
//     Q-buffer becomes value page E/G - 1; when L - R >= S, token L - R leaves
//     the local window for value Q-buffer slot (L - R - S) % G;
//   * token L goes to the sink (L < S) or to key Q-buffer slot (L - S) % G
//     and local window slot L % R.
// ---------------------------------------------------------------------------
struct AppendKittyParams {
    const int32_t *seq_len;
    const uint16_t *k_new, *v_new;
    uint8_t *k_pages, *v_pages;
    uint16_t *k_sink, *v_sink, *k_qbuf, *v_qbuf, *v_local;
    unsigned *err;
    int Hkv, S, R, K, score_mode, max_seq_len, page_cap;
    int64_t kpb, vpb;
    const int32_t *page_table;   // paged cache: pools [n_pages][Hkv][record]; null: per-request arrays
    int n_pages;
};

// Record index of logical page p of (row b, kv head h): per-request arrays,
// or the pool page of the page table (-1, KVQ_DEVICE_ERR_POOL recorded, for
// an entry outside the pool).
__device__ __forceinline__ int64_t kitty_record(const AppendKittyParams &P, int b, int h, int p) {
    if (!P.page_table) return ((int64_t)b * P.Hkv + h) * P.page_cap + p;
    const int pg = P.page_table[(int64_t)b * P.page_cap + p];
    if (pg < 0 || pg >= P.n_pages) {
        if (threadIdx.x == 0) atomicOr(P.err, KVQ_DEVICE_ERR_POOL);
        return -1;
    }
    return (int64_t)pg * P.Hkv + h;
}

__global__ void __launch_bounds__(128) append_kitty_kernel(AppendKittyParams P) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    constexpr int G = 128;
    const int64_t bk = blockIdx.x;
    const int b = (int)(bk / P.Hkv);
    const int L = P.seq_len[b];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (L < 0 || L >= P.max_seq_len) {
        if (threadIdx.x == 0) atomicOr(P.err, KVQ_DEVICE_ERR_CAPACITY);
        return;
    }
    const int S = P.S, R = P.R;
    const int h = (int)(bk - (int64_t)b * P.Hkv);
    // paged: a row whose next page could not be allocated is left unchanged
    if (P.page_table && L >= S && (L - S) % G == 0 && P.page_table[(int64_t)b * P.page_cap + (L - S) / G] < 0) return;
    uint16_t *kqb = P.k_qbuf + bk * G * KVQ_D;
    uint16_t *vqb = P.v_qbuf + bk * G * KVQ_D;
    uint16_t *vloc = P.v_local + bk * (int64_t)R * KVQ_D;
    if (L > S && (L - S) % G == 0) {
        const int64_t rec = kitty_record(P, b, h, (L - S) / G - 1);
        if (rec >= 0) kitty_key_page_quant<128>(kqb, P.K, P.score_mode, P.k_pages + rec * P.kpb, smem_raw);
    }
    const int E = L - S - R;
    const int64_t vrec = E > 0 && E % G == 0 ? kitty_record(P, b, h, E / G - 1) : -1;
    if (vrec >= 0) {
        uint8_t *pg = P.v_pages + vrec * P.vpb;
        uint16_t *ps = reinterpret_cast<uint16_t *>(pg + (int64_t)G * KVQ_D / 4);
        for (int tt = warp; tt < G; tt += 4) {
            uint32_t wv;
            uint16_t sv, zv;
            value_token_quant<128>(vqb + (int64_t)tt * KVQ_D, lane, wv, sv, zv);
            if ((lane & 3) == 0) reinterpret_cast<uint32_t *>(pg + (int64_t)tt * (KVQ_D / 4))[lane >> 2] = wv;
            if (lane == 0) {
                ps[tt] = sv;
                ps[G + tt] = zv;
            }
        }
    }
    __syncthreads();
    if (L - R >= S && threadIdx.x < 16) {
        const int te = L - R;
        reinterpret_cast<uint4 *>(vqb + (int64_t)((te - S) % G) * KVQ_D)[threadIdx.x] =
            reinterpret_cast<const uint4 *>(vloc + (int64_t)(te % R) * KVQ_D)[threadIdx.x];
    }
    __syncthreads();
    const uint4 *kn = reinterpret_cast<const uint4 *>(P.k_new + bk * KVQ_D);
    const uint4 *vn = reinterpret_cast<const uint4 *>(P.v_new + bk * KVQ_D);
    if (L < S) {
        if (threadIdx.x < 16)
            reinterpret_cast<uint4 *>(P.k_sink + (bk * S + L) * KVQ_D)[threadIdx.x] = kn[threadIdx.x];
        else if (threadIdx.x < 32)
            reinterpret_cast<uint4 *>(P.v_sink + (bk * S + L) * KVQ_D)[threadIdx.x - 16] = vn[threadIdx.x - 16];
    } else {
        if (threadIdx.x < 16)
            reinterpret_cast<uint4 *>(kqb + (int64_t)((L - S) % G) * KVQ_D)[threadIdx.x] = kn[threadIdx.x];
        else if (threadIdx.x < 32)
            reinterpret_cast<uint4 *>(vloc + (int64_t)(L % R) * KVQ_D)[threadIdx.x - 16] = vn[threadIdx.x - 16];
    }
}

static cudaError_t launch_append_kitty_impl(const kvq_config *cfg, const kvq_kitty_cache *c, const kvq_slot_pool *pool,
                                           const void *k_new, const void *v_new, int score_mode, cudaStream_t st) {
    AppendKittyParams P;
    P.seq_len = c->seq_len;
    P.k_new = static_cast<const uint16_t *>(k_new);
    P.v_new = static_cast<const uint16_t *>(v_new);
    P.k_pages = static_cast<uint8_t *>(const_cast<void *>(c->k_pages));
    P.v_pages = static_cast<uint8_t *>(const_cast<void *>(c->v_pages));
    P.k_sink = static_cast<uint16_t *>(const_cast<void *>(c->k_sink));
    P.v_sink = static_cast<uint16_t *>(const_cast<void *>(c->v_sink));
    P.k_qbuf = static_cast<uint16_t *>(const_cast<void *>(c->k_qbuf));
    P.v_qbuf = static_cast<uint16_t *>(const_cast<void *>(c->v_qbuf));
    P.v_local = static_cast<uint16_t *>(const_cast<void *>(c->v_local));
    P.err = device_error_ptr();
    if (!P.err) return cudaErrorInvalidDevicePointer;
    P.Hkv = cfg->n_kv_heads;
    P.S = cfg->sink;
    P.R = cfg->residual;
    P.K = cfg->boost_k;
    P.score_mode = score_mode;
    P.page_table = c->page_table;
    P.n_pages = c->n_pages;
    P.max_seq_len = c->max_seq_len;
    P.page_cap = (int)((c->max_seq_len - cfg->sink > 0 ? c->max_seq_len - cfg->sink : 0) + 127) / 128;
    if (P.page_cap < 1) P.page_cap = 1;
    P.kpb = kitty_key_page_bytes(cfg->boost_k);
    P.vpb = 128LL * KVQ_D / 4 + 4LL * 128;
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(append_kitty_kernel, KITTY_KEY_SMEM, attr_done)) return e;
    if (c->page_table) {
        cudaError_t e = launch_alloc_ids(c->seq_len, const_cast<int32_t *>(c->page_table), c->batch, c->max_seq_len,
                                         128, P.page_cap, cfg->sink, pool, st);
        if (e != cudaSuccess) return e;
    }
    append_kitty_kernel<<<(unsigned)((int64_t)c->batch * cfg->n_kv_heads), 128, KITTY_KEY_SMEM, st>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (c->page_table)
        append_bump_paged_kernel<<<(c->batch + 127) / 128, 128, 0, st>>>(
            const_cast<int32_t *>(c->seq_len), c->page_table, P.page_cap, cfg->sink, c->batch, c->max_seq_len);
    else
        append_bump_kernel<<<(c->batch + 127) / 128, 128, 0, st>>>(const_cast<int32_t *>(c->seq_len), c->batch,
                                                                    c->max_seq_len);
    return cudaGetLastError();
}

cudaError_t launch_append_kitty_paged(const kvq_config *cfg, const kvq_kitty_cache *c, const kvq_slot_pool *pool,
                                      const void *k_new, const void *v_new, int score_mode, cudaStream_t st) {
    return launch_append_kitty_impl(cfg, c, pool, k_new, v_new, score_mode, st);
}

cudaError_t launch_append_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *k_new, const void *v_new,
                                int score_mode, cudaStream_t st) {
    return launch_append_kitty_impl(cfg, c, nullptr, k_new, v_new, score_mode, st);
}

cudaError_t launch_philox(const uint32_t *ctr, const uint32_t *key, int64_t n, uint32_t *out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int grid = grid_cap((n + 255) / 256, 8);
    philox_kernel<<<grid, 256, 0, st>>>(ctr, key, n, out);
    return cudaGetLastError();
}

}  // namespace kvq
