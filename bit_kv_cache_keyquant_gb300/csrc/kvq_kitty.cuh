// Shared pieces of the Kitty decode kernels (a7): parameters, work units,
// the residual-token path and the producer warp.
#pragma once

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int NCWARP = 4;
constexpr int PG = 128;                    // tokens per page
constexpr int STAGE_BYTES = 12288;
constexpr int VREC_OFF = 7680;             // value record offset inside a stage (key record <= 7680 B)
constexpr int KMAX = 92;                   // boosted channels that fit the key-record slot

struct Params {
    const int32_t *seq_len;
    const uint8_t *k_pages;
    const uint8_t *v_pages;
    const uint16_t *k_sink, *v_sink, *k_qbuf, *v_qbuf, *v_local;
    const uint16_t *q;
    float *ws_o, *ws_lse;
    unsigned *err;
    int B, Hq, Hkv, S, R, K, splits, chunk, page_cap;
    int max_len;        // max_seq_len: seq_len[b] is read clamped into [0, max_len]
    int vsub;           // grouped-query units per kv head (each takes Hq / Hkv / vsub query heads)
    int gall, gu;       // query heads per kv head; per grouped-query unit (gall / vsub)
    int kpb, vpb;
    float alpha;
    int e0;
    // paged cache (page_table non-null): logical page p of row b is pool page
    // page_table[b * page_cap + p] of k_pages / v_pages ([n_pages][Hkv][record])
    const int32_t *page_table;
    int n_pages;
};

struct Unit {
    int b, hq, kvh, sub, split, p0, np, nKp, nVp, nkb, nvb, L;
    bool residual;
    int64_t bk;
};

// hpr = units per batch row and split: P.Hq (one query head per unit) or
// P.Hkv (all query heads of a kv head per unit; hq is then the kv head).
// Row-major (u = row * splits + split) or split-major (u = split * rows +
// row: every CTA's round-robin share mixes all splits; used by the
// grouped-query kernel's long units).
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
    U.L = L;
    if (L > P.S) {
        U.nkb = ((L - P.S - 1) % PG) + 1;
        U.nKp = (L - P.S - U.nkb) / PG;
    } else {
        U.nkb = 0;
        U.nKp = 0;
    }
    const int E = max(0, L - P.S - P.R);
    U.nvb = E > 0 ? ((E - 1) % PG) + 1 : 0;
    U.nVp = (E - U.nvb) / PG;
    const int Pf = min(U.nKp, U.nVp);                  // pages quantized on both sides
    U.residual = U.split == P.splits - 1;
    if (U.residual) {
        U.p0 = Pf;
        U.np = 0;
    } else {
        const int cpp = P.chunk / PG;
        U.p0 = U.split * cpp;
        U.np = max(0, min(U.p0 + cpp, Pf) - U.p0);
    }
    const int upk = hpr / P.Hkv;                       // units per kv head: Hq / Hkv, or vsub
    U.kvh = U.hq / upk;
    U.sub = U.hq - U.kvh * upk;
    U.bk = (int64_t)U.b * P.Hkv + U.kvh;
    return U;
}

// Record index of logical page p of the unit's (row, kv head): the dense
// per-request arrays, or the pool page the page table names (an entry
// outside the pool reads page 0 and records KVQ_DEVICE_ERR_POOL).
__device__ __forceinline__ int64_t page_record(const Params &P, const Unit &U, int p) {
    if (!P.page_table) return U.bk * P.page_cap + p;
    int pg = P.page_table[(int64_t)U.b * P.page_cap + p];
    if (pg < 0 || pg >= P.n_pages) {
        atomicOr(P.err, KVQ_DEVICE_ERR_POOL);
        pg = 0;
    }
    return (int64_t)pg * P.Hkv + U.kvh;
}

__device__ __forceinline__ const uint8_t *key_page(const Params &P, const Unit &U, int p) {
    return P.k_pages + page_record(P, U, p) * (int64_t)P.kpb;
}

__device__ __forceinline__ const uint8_t *value_page(const Params &P, const Unit &U, int p) {
    return P.v_pages + page_record(P, U, p) * (int64_t)P.vpb;
}

// Byte of token tt (0..127) of a key page's planes, bit position 2 * ((tt % 32) / 8):
// the low plane in the KIVI 2-bit key-tile order (channel c = 16k + 2r + e + 8h of
// token q + 8p of tile j at byte j*1024 + (k/4)*512 + (4q + r)*16 + (k%4)*4 + e + 2h),
// the high plane in blocks of kp * 8 bytes per 32-token tile (row 16kh + 4rb + b at
// byte 128kh + 32rb + 4q + b of its tile's block; kp = the plane's rows).
__device__ __forceinline__ int kitty_low_byte(int tt, int c) {
    const int q = tt & 7, k = c >> 4, cc = c & 15;
    return (tt >> 5) * 1024 + (k >> 2) * 512 + (4 * q + ((cc & 7) >> 1)) * 16 + (k & 3) * 4 + (cc & 1) + 2 * (cc >> 3);
}
__device__ __forceinline__ int kitty_high_byte(int kp, int tt, int row) {
    return (tt >> 5) * 8 * kp + (row >> 4) * 128 + ((row & 15) >> 2) * 32 + 4 * (tt & 7) + (row & 3);
}

// Tokens of one query head outside whole pages (sink, Q-buffers, local
// window, a key page whose values are still fp16): lane = token for the keys
// (independent per-lane loads), four channels per lane for the values.
// qv = alpha q of the head (shared memory, channel order).
__device__ __forceinline__ void kitty_residual(const Params &P, const Unit &U, const float *qv, int warp, int lane,
                                               float racc[4], float &m_run, float &l_part) {
    const int K = P.K;
    const int nA = min(U.L, P.S);
    const int tB = P.S + U.p0 * PG;
    const int nB = max(0, U.L - tB);
    const int ntok = nA + nB;
    m_run = -INFINITY;
    l_part = 0.f;
    racc[0] = racc[1] = racc[2] = racc[3] = 0.f;
    const uint16_t *ksink = P.k_sink + U.bk * (int64_t)P.S * KVQ_D;
    const uint16_t *vsink = P.v_sink + U.bk * (int64_t)P.S * KVQ_D;
    const uint16_t *kqb = P.k_qbuf + U.bk * (int64_t)PG * KVQ_D;
    const uint16_t *vqb = P.v_qbuf + U.bk * (int64_t)PG * KVQ_D;
    const uint16_t *vloc = P.v_local + U.bk * (int64_t)P.R * KVQ_D;
    const int vq_end = P.S + U.nVp * PG + U.nvb;           // value Q-buffer tokens end here
    for (int i0 = 32 * warp; i0 < ntok; i0 += 32 * NCWARP) {
        const int n = min(32, ntok - i0);
        // ---- keys: lane = token ----
        const int i = i0 + min(lane, n - 1);
        const int t = i < nA ? i : tB + (i - nA);
        float logit = 0.f;
        if (t < P.S || t >= P.S + U.nKp * PG) {
            const uint16_t *row = t < P.S ? ksink + (int64_t)t * KVQ_D : kqb + (int64_t)((t - P.S) % PG) * KVQ_D;
#pragma unroll 4
            for (int c8 = 0; c8 < 16; ++c8) {
                const uint4 u4 = __ldg(reinterpret_cast<const uint4 *>(row) + c8);
                const float4 qa0 = *reinterpret_cast<const float4 *>(&qv[8 * c8]);
                const float4 qa1 = *reinterpret_cast<const float4 *>(&qv[8 * c8 + 4]);
                logit += qa0.x * h2f(lo16(u4.x)) + qa0.y * h2f(hi16(u4.x)) + qa0.z * h2f(lo16(u4.y)) +
                         qa0.w * h2f(hi16(u4.y)) + qa1.x * h2f(lo16(u4.z)) + qa1.y * h2f(hi16(u4.z)) +
                         qa1.z * h2f(lo16(u4.w)) + qa1.w * h2f(hi16(u4.w));
            }
        } else {
            const int p = (t - P.S) / PG, tt = (t - P.S) % PG;
            const uint8_t *pg = key_page(P, U, p);
            const int kp = kitty_high_rows(K), sh = 2 * ((tt & 31) >> 3);
            const uint8_t *low = pg, *high = pg + KVQ_D * PG / 4, *idx = high + (int64_t)kp * PG / 4;
            const uint16_t *ps = reinterpret_cast<const uint16_t *>(idx + KVQ_D);
            for (int c = 0; c < KVQ_D; ++c) {
                int code = (low[kitty_low_byte(tt, c)] >> sh) & 3;
                const int r = idx[c];
                if (r < K) code |= ((high[kitty_high_byte(kp, tt, r)] >> sh) & 3) << 2;
                logit += qv[c] * ((float)code * h2f(ps[c]) + h2f(ps[KVQ_D + c]));
            }
        }
        if (lane >= n) logit = -INFINITY;
        const float mt = warp_max(logit);
        if (mt > m_run) {
            const float sc = exp2f(m_run - mt);
            l_part *= sc;
#pragma unroll
            for (int k = 0; k < 4; ++k) racc[k] *= sc;
            m_run = mt;
        }
        const float p = exp2f(logit - m_run);
        l_part += p;
        // ---- values: lane = channels 4*lane..4*lane+3; every value here is fp16 ----
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
            const int ij = i0 + min(j, n - 1);
            const int tj = ij < nA ? ij : tB + (ij - nA);
            const uint16_t *vrow = tj < P.S ? vsink + (int64_t)tj * KVQ_D
                                 : tj < vq_end ? vqb + (int64_t)((tj - P.S) % PG) * KVQ_D
                                               : vloc + (int64_t)(tj % P.R) * KVQ_D;
            const uint2 vv = __ldg(reinterpret_cast<const uint2 *>(vrow + 4 * lane));
            const float pj = __shfl_sync(0xFFFFFFFFu, p, j);        // 0 for j >= n
            racc[0] += pj * h2f(lo16(vv.x));
            racc[1] += pj * h2f(hi16(vv.x));
            racc[2] += pj * h2f(lo16(vv.y));
            racc[3] += pj * h2f(hi16(vv.y));
        }
    }
}

// Producer (one lane): one page (key record, value record) per stage, in
// unit order, into an NST-slot ring; returns after every issued copy landed.
template <int NST, bool SPLIT_MAJOR = false>
__device__ __forceinline__ void kitty_produce(const Params &P, int hpr, uint8_t (*stage)[STAGE_BYTES], uint64_t *full,
                                              uint64_t *empty, const int *abort_flag) {
    const int n_units = P.B * hpr * P.splits;
    bool ok = true;
    int sg = 0;
    int armed[NST];
#pragma unroll
    for (int j = 0; j < NST; ++j) armed[j] = 0;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const Unit U = unit_of<SPLIT_MAJOR>(P, u, hpr);
        for (int s = 0; s < U.np; ++s, ++sg) {
            const int slot = sg % NST;
            if (sg >= NST) ok = mbar_wait(&empty[slot], ((sg / NST) - 1) & 1, P.err);
            ok = ok && !ring_aborted(abort_flag);
            if (!ok) break;
            const int p = U.p0 + s;
            uint8_t *st = stage[slot];
            ++armed[slot];
            mbar_expect_tx(&full[slot], (uint32_t)(P.kpb + P.vpb));
            bulk_g2s(st, key_page(P, U, p), (uint32_t)P.kpb, &full[slot]);
            bulk_g2s(st + VREC_OFF, value_page(P, U, p), (uint32_t)P.vpb, &full[slot]);
        }
    }
    producer_drain<NST>(full, armed, P.err);
}

}  // namespace
}  // namespace kvq
