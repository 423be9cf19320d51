// Shared pieces of the KIVI decode kernels (a3): parameters, work units,
// the packed-key addressing, fallback element fetches and the producer
// warp that streams 128-token stages with bulk async copies.
#pragma once

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int NCWARP = 4;                 // consumer warps
constexpr int STAGE_TOK = 32 * NCWARP;    // 128 tokens per stage
constexpr int KC_BYTES = STAGE_TOK * KVQ_D / 4;        // 4096
constexpr int KSZ_MAX = 4 * KVQ_D * 4;                  // 2048 (G = 32)
constexpr int VC_BYTES = STAGE_TOK * KVQ_D / 4;        // 4096
constexpr int VSZ_MAX = STAGE_TOK * 4 * 4;             // 2048 (Gv = 32)
constexpr int STAGE_BYTES = KC_BYTES + KSZ_MAX + VC_BYTES + VSZ_MAX;   // 12288

// Stage geometry for BK-bit keys and BV-bit values (2 or 4): key codes, key
// (s, z), value codes, value (s, z), in that order.
template <int BK, int BV>
struct Geo {
    static constexpr int KC = STAGE_TOK * KVQ_D * BK / 8;
    static constexpr int KSZ = KSZ_MAX;
    static constexpr int VC = STAGE_TOK * KVQ_D * BV / 8;
    static constexpr int VSZ = VSZ_MAX;
    static constexpr int BYTES = KC + KSZ + VC + VSZ;
};
static_assert(Geo<2, 2>::BYTES == STAGE_BYTES, "2-bit stage geometry");

struct Params {
    const int32_t *seq_len;
    const uint8_t *k_codes;
    const uint32_t *k_sz;
    const uint8_t *v_codes;
    const uint32_t *v_sz;
    const uint16_t *k_res;
    const uint16_t *v_res;
    const uint16_t *q;
    float *ws_o;
    float *ws_lse;
    unsigned *err;
    int B, Hq, Hkv, G, Gv, R, splits, chunk;
    int ngv;            // D / Gv: value (s, z) pairs per token
    int vsub;           // grouped-query units per kv head (each takes Hq / Hkv / vsub query heads)
    int gall, gu;       // query heads per kv head; per grouped-query unit (gall / vsub)
    int max_len;        // max_seq_len: seq_len[b] is read clamped into [0, max_len]
    int64_t cap;        // token capacity per (b, kvh): max_seq_len rounded up to 128
    int64_t kgrp_cap;   // cap / G
    float alpha;
    int bits_k, bits_v; // code widths (2 or 4)
    int vtiles;         // values stored in value tiles (kivi_value_tiles), else token-major
    // paged cache (page_table non-null): token t of row b is in page record
    // pages + (page_table[b * pt_stride + t / 128] * Hkv + kv head) * rec_bytes
    const int32_t *page_table;
    const uint8_t *pages;
    int pt_stride, n_pages;
    int64_t rec_bytes;
    int kc_bytes, vc_bytes;   // page record sections: key codes, key (s, z) (2048 B), value codes, value (s, z)
#ifdef KVQ_FAULT_INJECT
    int inj_skip;             // test builds: stage of CTA 0 the producer leaves unfilled (-1: none)
    unsigned inj_spin;        // test builds: wait tries before giving up (0: KVQ_SPIN_LIMIT)
#endif
};

// Tries of a bounded mbarrier wait in the KIVI decode kernels.
#ifdef KVQ_FAULT_INJECT
#define KIVI_WAIT_LIMIT(P) ((P).inj_spin ? (P).inj_spin : KVQ_SPIN_LIMIT)
#else
#define KIVI_WAIT_LIMIT(P) KVQ_SPIN_LIMIT
#endif

// Geometry of one work unit.  Splits 0 .. splits-2 of a (batch row, query
// head) cover the staged quantized tiles [0, Qf) in chunks; split splits-1
// covers every remaining token [Qf, L) (the fp16 residual and any tokens cut
// off by a segment boundary), read straight from global memory.
struct Unit {
    int b, hq, kvh, sub, split, t0, t1, nT, nstages, nKq, nVq;
    bool residual;
    int64_t bk;
};

// hpr = units per batch row and split: P.Hq (one query head per unit) or
// P.Hkv * P.vsub (a kv head's query heads in vsub units; hq then indexes
// (kv head, sub)).
// Units are numbered row-major (u = row * splits + split) or, for the long
// units of the grouped-query kernels, split-major (u = split * rows + row),
// which gives every CTA's round-robin share a mix of all splits (measured:
// 4.5% faster on the grouped-query workload; the per-head kernel is faster
// row-major).
template <bool SPLIT_MAJOR = false>
__device__ __forceinline__ Unit unit_of(const Params &P, int u, int hpr) {
    Unit U;
    int row;
    if (SPLIT_MAJOR) {
        const int rows = P.B * hpr;
        U.split = u / rows;
        row = u - U.split * rows;
    } else {
        row = u / P.splits;
        U.split = u - row * P.splits;
    }
    U.b = row / hpr;
    U.hq = row - U.b * hpr;
    const int L = clamp_len(P.seq_len[U.b], P.max_len, P.err);
    const int rK = ((L - 1) % P.R) + 1;
    U.nKq = L - rK;
    U.nVq = L - (L < P.R ? L : P.R);
    const int Qf = (U.nKq < U.nVq ? U.nKq : U.nVq) & ~31;
    U.residual = U.split == P.splits - 1;
    if (U.residual) {
        U.t0 = Qf;
        U.t1 = L;
        U.nT = 0;
    } else {
        U.t0 = U.split * P.chunk;
        U.t1 = max(U.t0, min(U.t0 + P.chunk, Qf));
        U.nT = (U.t1 - U.t0) / 32;
    }
    U.nstages = (U.nT + NCWARP - 1) / NCWARP;
    const int upk = hpr / P.Hkv;                       // units per kv head: Hq / Hkv, or vsub
    U.kvh = U.hq / upk;
    U.sub = U.hq - U.kvh * upk;
    U.bk = (int64_t)U.b * P.Hkv + U.kvh;
    return U;
}

// Page record holding token t of the unit's (row, kv head) in a paged cache;
// a table entry outside the pool reads page 0 and records KVQ_DEVICE_ERR_POOL.
__device__ __forceinline__ const uint8_t *kivi_page(const Params &P, const Unit &U, int t) {
    int pg = P.page_table[(int64_t)U.b * P.pt_stride + (t >> 7)];
    if (pg < 0 || pg >= P.n_pages) {
        atomicOr(P.err, KVQ_DEVICE_ERR_POOL);
        pg = 0;
    }
    return P.pages + ((int64_t)pg * P.Hkv + U.kvh) * P.rec_bytes;
}

// KIVI key storage (see kv_quant_key): token t = q + 8p, channel c = 16k + cc
// with cc = 2r + e + 8h sits in bits 2p of byte e + 2h of word k%4 of chunk
// 4q + r of half k/4 of its 32-token tile; the group's (s, z) block is 128
// fp16 scales then 128 fp16 zeros at ((k/2)*4 + r)*8 + (k%2)*4 + e + 2h.
__device__ __forceinline__ int kivi_key_byte_offset(int t, int c) {
    const int k = c >> 4, cc = c & 15;
    return (t >> 5) * 1024 + (k >> 2) * 512 + (4 * (t & 7) + ((cc & 7) >> 1)) * 16 + (k & 3) * 4 + (cc & 1) +
           2 * (cc >> 3);
}

// The same layout at b bits: a 32-token tile is b/2 planes of 1024 bytes and
// token q + 8p sits in plane p / (8/b) at bits b * (p % (8/b)).
__device__ __forceinline__ int kivi_key_byte_offset_w(int bits, int t, int c) {
    const int cpb = 8 / bits, p = (t & 31) >> 3;
    return (t >> 5) * 512 * bits + (p / cpb) * 1024 + kivi_key_byte_offset(t & 7, c);
}

__device__ __forceinline__ int kivi_key_bit_w(int bits, int t) { return bits * (((t & 31) >> 3) % (8 / bits)); }

__device__ __forceinline__ int kivi_sz_index(int c) {
    const int k = c >> 4, cc = c & 15;
    return ((k >> 1) * 4 + ((cc & 7) >> 1)) * 8 + (k & 1) * 4 + (cc & 1) + 2 * (cc >> 3);
}

// Four dequantized key / value channels 4*lane..4*lane+3 of token t, from the
// quantized segment or the fp16 residual (used outside the staged tiles).
__device__ __forceinline__ void fetch_k4(const Params &P, const Unit &U, int t, int lane, float kv[4]) {
    if (t < U.nKq) {
        const int G = P.G, gi = t / G, tt = t - gi * G;
        const int bits = P.bits_k;
        const uint8_t *grp;
        const uint16_t *szb;
        if (P.page_table) {
            const uint8_t *rec = kivi_page(P, U, t);
            const int gp = (t & 127) / G;                       // group within the page
            grp = rec + gp * (G * KVQ_D * bits / 8);
            szb = reinterpret_cast<const uint16_t *>(rec + P.kc_bytes + gp * 512);
        } else {
            grp = P.k_codes + (U.bk * P.kgrp_cap + gi) * ((int64_t)G * KVQ_D * bits / 8);
            szb = reinterpret_cast<const uint16_t *>(P.k_sz + (U.bk * P.kgrp_cap + gi) * KVQ_D);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = 4 * lane + i, si = kivi_sz_index(c);
            const int code = (grp[kivi_key_byte_offset_w(bits, tt, c)] >> kivi_key_bit_w(bits, tt)) & ((1 << bits) - 1);
            kv[i] = (float)code * h2f(szb[si]) + h2f(szb[KVQ_D + si]);
        }
    } else {
        const uint2 u = *reinterpret_cast<const uint2 *>(P.k_res + (U.bk * P.R + t % P.R) * KVQ_D + 4 * lane);
        kv[0] = h2f(lo16(u.x)); kv[1] = h2f(hi16(u.x)); kv[2] = h2f(lo16(u.y)); kv[3] = h2f(hi16(u.y));
    }
}

__device__ __forceinline__ void fetch_v4(const Params &P, const Unit &U, int t, int lane, float vv[4]) {
    if (t < U.nVq) {
        // the lane's 4 channels: one byte at 2 bits, two at 4 bits (channel c at bits bits*(c % (8/bits)))
        const int bits = P.bits_v;
        // the byte (2 bits) or 16-bit word (4 bits) of channel quad `lane`: in the value tiles, or token-major
        const uint8_t *vb;
        const uint32_t *szr;
        int64_t tl;                                            // the token within vb's tiles or rows
        if (P.page_table) {
            const uint8_t *rec = kivi_page(P, U, t);
            tl = t & 127;
            vb = rec + P.kc_bytes + 2048;
            szr = reinterpret_cast<const uint32_t *>(rec + P.kc_bytes + 2048 + P.vc_bytes) + tl * P.ngv;
        } else {
            tl = t;
            vb = P.v_codes + U.bk * P.cap * (KVQ_D * bits / 8);
            szr = P.v_sz + (U.bk * P.cap + t) * P.ngv;
        }
        uint32_t w;
        if (P.vtiles && bits == 2) {
            w = vb[kivi_value_byte(tl, lane)];
        } else if (P.vtiles) {
            w = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) w |= ((uint32_t)(vb[kivi_value_byte4(tl, 4 * lane + i)] >> (4 * (lane >> 4))) & 15u) << (4 * i);
        } else {
            w = bits == 2 ? (uint32_t)vb[tl * (KVQ_D / 4) + lane]
                          : (uint32_t)reinterpret_cast<const uint16_t *>(vb + tl * (KVQ_D / 2))[lane];
        }
        const uint32_t sz = szr[(4 * lane) / P.Gv];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            vv[i] = (float)((w >> (bits * i)) & ((1u << bits) - 1)) * h2f(lo16(sz)) + h2f(hi16(sz));
    } else {
        const uint2 u = *reinterpret_cast<const uint2 *>(P.v_res + (U.bk * P.R + t % P.R) * KVQ_D + 4 * lane);
        vv[0] = h2f(lo16(u.x)); vv[1] = h2f(hi16(u.x)); vv[2] = h2f(lo16(u.y)); vv[3] = h2f(hi16(u.y));
    }
}

// Residual unit of one query head (tokens [U.t0, U.t1) outside the staged
// tiles): 32 tokens per warp, lane = token for the logits, every load of a
// block issued together; lane l accumulates output channels 4l..4l+3.
__device__ __forceinline__ void kivi_residual(const Params &P, const Unit &U, const float qa[4], int warp, int lane,
                                              float racc[4], float &m_run, float &l_part) {
    m_run = -INFINITY;
    l_part = 0.f;
    racc[0] = racc[1] = racc[2] = racc[3] = 0.f;
    for (int r0 = U.t0 + 32 * warp; r0 < U.t1; r0 += 32 * NCWARP) {
        const int n = min(32, U.t1 - r0);
        // whole block fp16 in both K and V (the usual case): unconditional loads,
        // 8 tokens in flight per batch; indices clamped into the block
        const bool plain = r0 >= U.nKq && r0 >= U.nVq;
        const uint16_t *kres = P.k_res + U.bk * P.R * KVQ_D + 4 * lane;
        const uint16_t *vres = P.v_res + U.bk * P.R * KVQ_D + 4 * lane;
        float d[32];
        if (plain) {
#pragma unroll
            for (int hb = 0; hb < 4; ++hb) {
                uint2 raw[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int t = min(r0 + 8 * hb + m, U.t1 - 1);
                    raw[m] = __ldg(reinterpret_cast<const uint2 *>(kres + (t % P.R) * KVQ_D));
                }
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    d[8 * hb + m] = qa[0] * h2f(lo16(raw[m].x)) + qa[1] * h2f(hi16(raw[m].x)) +
                                     qa[2] * h2f(lo16(raw[m].y)) + qa[3] * h2f(hi16(raw[m].y));
            }
        } else {
#pragma unroll
            for (int tt = 0; tt < 32; ++tt) {
                d[tt] = 0.f;
                if (tt < n) {
                    float kv[4];
                    fetch_k4(P, U, r0 + tt, lane, kv);
                    d[tt] = qa[0] * kv[0] + qa[1] * kv[1] + qa[2] * kv[2] + qa[3] * kv[3];
                }
            }
        }
        // reduce-scatter over all 32 lanes: lane keeps token (bit-reversed lane index)
#pragma unroll
        for (int o = 16, h = 16; o >= 1; o >>= 1, h >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int m = 0; m < h; ++m) {
                const float send = up ? d[m] : d[m + h];
                d[m] = (up ? d[m + h] : d[m]) + __shfl_xor_sync(0xFFFFFFFFu, send, o);
            }
        }
        // lane holds token 16*b4 + 8*b3 + 4*b2 + 2*b1 + b0 = lane
        const float logit = lane < n ? d[0] : -INFINITY;
        const float mt = warp_max(logit);
        if (mt > m_run) {
            const float sc = exp2f(m_run - mt);
            l_part *= sc;
#pragma unroll
            for (int i = 0; i < 4; ++i) racc[i] *= sc;
            m_run = mt;
        }
        const float p = exp2f(logit - m_run);
        l_part += p;
        if (plain) {
#pragma unroll
            for (int hb = 0; hb < 4; ++hb) {
                uint2 raw[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int t = min(r0 + 8 * hb + m, U.t1 - 1);
                    raw[m] = __ldg(reinterpret_cast<const uint2 *>(vres + (t % P.R) * KVQ_D));
                }
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float pt = __shfl_sync(0xFFFFFFFFu, p, 8 * hb + m);   // 0 beyond the block
                    racc[0] += pt * h2f(lo16(raw[m].x));
                    racc[1] += pt * h2f(hi16(raw[m].x));
                    racc[2] += pt * h2f(lo16(raw[m].y));
                    racc[3] += pt * h2f(hi16(raw[m].y));
                }
            }
        } else {
#pragma unroll 1
            for (int tt = 0; tt < n; ++tt) {
                const float pt = __shfl_sync(0xFFFFFFFFu, p, tt);
                float vv[4];
                fetch_v4(P, U, r0 + tt, lane, vv);
#pragma unroll
                for (int i = 0; i < 4; ++i) racc[i] += pt * vv[i];
            }
        }
    }
}

// Producer (one lane): streams the stages of every unit of this CTA, in
// unit order, into an NST-slot ring; returns after every issued copy landed.
template <int NST, bool SPLIT_MAJOR = false, int BK = 2, int BV = 2>
__device__ __forceinline__ void kivi_produce(const Params &P, int hpr, uint8_t (*stage)[Geo<BK, BV>::BYTES],
                                             uint64_t *full, uint64_t *empty, const int *abort_flag) {
    using GG = Geo<BK, BV>;
    const int n_units = P.B * hpr * P.splits;
    const int G = P.G;
    bool ok = true;
    int sg = 0;
    int armed[NST];
#pragma unroll
    for (int j = 0; j < NST; ++j) armed[j] = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit U = unit_of<SPLIT_MAJOR>(P, u, hpr);
        const uint8_t *kc_base = P.k_codes + U.bk * P.kgrp_cap * ((int64_t)G * KVQ_D * BK / 8);
        const uint32_t *ksz_base = P.k_sz + U.bk * P.kgrp_cap * KVQ_D;
        const uint8_t *vc_base = P.v_codes + U.bk * P.cap * (KVQ_D * BV / 8);
        const uint32_t *vsz_base = P.v_sz + U.bk * P.cap * P.ngv;
        for (int s = 0; s < U.nstages; ++s, ++sg) {
            const int slot = sg % NST;
            if (sg >= NST) ok = mbar_wait(&empty[slot], ((sg / NST) - 1) & 1, P.err, KIVI_WAIT_LIMIT(P));
            ok = ok && !ring_aborted(abort_flag);
            if (!ok) break;
#ifdef KVQ_FAULT_INJECT
            if (blockIdx.x == 0 && sg == P.inj_skip) continue;   // test builds: this stage never fills
#endif
            const int nt = min(NCWARP, U.nT - s * NCWARP);
            const int tok = U.t0 + s * STAGE_TOK;
            const uint32_t kc_b = nt * 512 * BK;
            const uint32_t ksz_b = ((nt * 32 + G - 1) / G) * KVQ_D * 4;
            const uint32_t vc_b = nt * 32 * (KVQ_D * BV / 8);
            const uint32_t vsz_b = nt * 32 * P.ngv * 4;
            uint8_t *st = stage[slot];
            ++armed[slot];
            if (P.page_table) {
                // the page record is the stage: one copy (the tiles past nt are not read)
                mbar_expect_tx(&full[slot], (uint32_t)GG::BYTES);
                bulk_g2s(st, kivi_page(P, U, tok), (uint32_t)GG::BYTES, &full[slot]);
                continue;
            }
            mbar_expect_tx(&full[slot], kc_b + ksz_b + vc_b + vsz_b);
            bulk_g2s(st, kc_base + (int64_t)(tok >> 5) * 512 * BK, kc_b, &full[slot]);
            bulk_g2s(st + GG::KC, ksz_base + (int64_t)(tok / G) * KVQ_D, ksz_b, &full[slot]);
            bulk_g2s(st + GG::KC + GG::KSZ, vc_base + (int64_t)tok * (KVQ_D * BV / 8), vc_b, &full[slot]);
            bulk_g2s(st + GG::KC + GG::KSZ + GG::VC, vsz_base + (int64_t)tok * P.ngv, vsz_b, &full[slot]);
        }
    }
    // drain: every issued copy must have landed before the CTA exits
    producer_drain<NST>(full, armed, P.err, KIVI_WAIT_LIMIT(P));
}

// Kernel parameters common to the KIVI decode kernels, from a dense or paged cache.
inline Params kivi_params(const kvq_config *cfg, const KiviSrc &c, const void *q, const DecodePlan &p, void *ws) {
    Params P;
    P.seq_len = c.seq_len;
    P.k_codes = static_cast<const uint8_t *>(c.k_codes);
    P.k_sz = static_cast<const uint32_t *>(c.k_sz);
    P.v_codes = static_cast<const uint8_t *>(c.v_codes);
    P.v_sz = static_cast<const uint32_t *>(c.v_sz);
    P.k_res = static_cast<const uint16_t *>(c.k_res);
    P.v_res = static_cast<const uint16_t *>(c.v_res);
    P.q = static_cast<const uint16_t *>(q);
    P.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_o);
    P.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_lse);
    P.err = device_error_ptr();
    P.B = c.batch;
    P.Hq = cfg->n_q_heads;
    P.Hkv = cfg->n_kv_heads;
    P.G = cfg->group_k;
    P.Gv = cfg->group_v;
    P.ngv = KVQ_D / cfg->group_v;
    P.vsub = 1;
    P.gall = cfg->n_q_heads / cfg->n_kv_heads;
    P.gu = P.gall;
    P.R = cfg->residual;
    P.max_len = c.max_seq_len;
    P.cap = ((int64_t)c.max_seq_len + 127) / 128 * 128;
    P.splits = p.splits;
    P.chunk = p.chunk;
    P.kgrp_cap = P.cap / cfg->group_k;
    P.alpha = sm_scale_of(cfg) * 1.4426950408889634f;
    P.bits_k = cfg->bits_k;
    P.bits_v = cfg->bits_v;
    P.vtiles = kivi_value_tiles(cfg);
    P.page_table = c.page_table;
    P.pages = static_cast<const uint8_t *>(c.pages);
    P.pt_stride = (int)(P.cap / 128);
    P.n_pages = c.n_pages;
    P.rec_bytes = kivi_page_bytes(cfg->bits_k, cfg->bits_v);
    P.kc_bytes = 16 * KVQ_D * cfg->bits_k;
    P.vc_bytes = 16 * KVQ_D * cfg->bits_v;
#ifdef KVQ_FAULT_INJECT
    P.inj_skip = g_test_inject.skip_stage;
    P.inj_spin = g_test_inject.spin_limit;
#endif
    return P;
}

}  // namespace
}  // namespace kvq
