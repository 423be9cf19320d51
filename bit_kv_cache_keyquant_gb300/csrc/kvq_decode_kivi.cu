// a3: KIVI split-KV decode attention, stage 1 (one CTA per (split, query
// head, batch row)).
//
// Math (KIVI Eq. 3 with the dequantization folded out of the inner loops):
//   score_t = alpha * sum_c q_c (s_cg code_ct + z_cg)
//           = sum_c (alpha q_c s_cg) code_ct + alpha sum_c q_c z_cg
//   o_c     = sum_t p_t (s_tj code_tc + z_tj)
//           = sum_t (p_t s_tj) code_tc + sum_t p_t z_tj
// with alpha = sm_scale * log2(e) (softmax in base 2).
// Keys: a 2-bit code masked in place out of its packed word, read as an fp32
// bit pattern, is the denormal code * 2^(k-149) (k = its bit position, kept
// below the exponent field), so one LOP3 makes an exact fp32 operand and a
// packed fma.rn.f32x2 multiplies it by alpha q s pre-scaled by 2^(149-k-E0);
// every product is alpha q s code 2^(2j-E0), exact in fp32 (the fp32 weight
// matters: a logit error is amplified by the softmax).
// Values: the same masking read as fp16 subnormals (code * 2^(2i-24)), two
// codes per LOP3, accumulated by fma.rn.f32.f16 with the fp16 weight
// p_t s_tj (a weight's rounding is not amplified).
// Powers of two are removed once per token (keys) or channel (values).
//
// Data movement: a producer warp streams 128-token stages (key codes, key
// (s, z), value codes, value (s, z): 12 KiB at G = Gv = 32) with 1-D bulk
// async copies (cp.async.bulk, the TMA engine) into a 4-slot shared-memory
// ring guarded by mbarriers; four consumer warps each take one 32-token tile
// of a stage.  Tokens whose key or value is not quantized (the fp16
// residual) take a per-token path.  Each warp keeps its own online softmax
// state; the CTA merges the eight warp states and writes (o_s, lse_s).
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int NSTAGE = 4;
constexpr int NCWARP = 4;                 // consumer warps
constexpr int STAGE_TOK = 32 * NCWARP;    // 128 tokens per stage
constexpr int KC_BYTES = STAGE_TOK * KVQ_D / 4;        // 4096
constexpr int KSZ_MAX = 4 * KVQ_D * 4;                  // 2048 (G = 32)
constexpr int VC_BYTES = STAGE_TOK * KVQ_D / 4;        // 4096
constexpr int VSZ_MAX = STAGE_TOK * 4 * 4;             // 2048 (Gv = 32)
constexpr int STAGE_BYTES = KC_BYTES + KSZ_MAX + VC_BYTES + VSZ_MAX;   // 12288
constexpr int NSTATE = 2 * NCWARP;

struct Smem {
    uint8_t stage[NSTAGE][STAGE_BYTES];
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    float qk[NCWARP][KVQ_D];              // per-warp alpha*q*s*2^(149-8(c&1)-E0) of the current key group
    float st_acc[NSTATE][KVQ_D];
    float st_m[NSTATE];
    float st_l[NSTATE];
};

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
    int Hq, Hkv, G, Gv, R, splits, chunk;
    int64_t cap;        // token capacity per (b, kvh): max_seq_len rounded up to 128
    int64_t kgrp_cap;   // cap / G
    float alpha;
    int e0;             // product exponent offset: every key product is scaled by 2^-E0
};

__device__ __forceinline__ int kivi_key_byte_offset(int t, int c) {
    return (t >> 5) * 1024 + ((c >> 4) & 1) * 512 + (4 * ((t & 31) >> 2) + (c >> 5)) * 16 + ((c >> 2) & 3) * 4 + (c & 3);
}

}  // namespace

__global__ void __launch_bounds__(32 * (NCWARP + 1), 4) kivi_decode_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>(smem_raw);
    const int split = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
    const int g = P.Hq / P.Hkv;
    const int kvh = hq / g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = P.seq_len[b];
    const int R = P.R, G = P.G, Gv = P.Gv;
    const int rK = ((L - 1) % R) + 1;
    const int nKq = L - rK;
    const int nVq = L - (L < R ? L : R);
    const int Qf = (nKq < nVq ? nKq : nVq) & ~31;         // fast tiles end here
    const int t0 = split * P.chunk;
    const int t1 = min(t0 + P.chunk, L);
    const int fast_end = max(t0, min(t1, Qf));
    const int nT = (fast_end - t0) / 32;                  // full 32-token tiles
    const int nstages = (nT + NCWARP - 1) / NCWARP;
    const int64_t bk = (int64_t)b * P.Hkv + kvh;
    const uint8_t *kc_base = P.k_codes + bk * P.kgrp_cap * ((int64_t)G * KVQ_D / 4);
    const uint32_t *ksz_base = P.k_sz + bk * P.kgrp_cap * KVQ_D;
    const uint8_t *vc_base = P.v_codes + bk * P.cap * (KVQ_D / 4);
    const uint32_t *vsz_base = P.v_sz + bk * P.cap * (KVQ_D / Gv);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], NCWARP);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCWARP) {
        // ---------------- producer ----------------
        if (lane == 0) {
            bool ok = true;
            for (int s = 0; s < nstages && ok; ++s) {
                const int slot = s % NSTAGE;
                if (s >= NSTAGE) ok = mbar_wait(&S.empty[slot], ((s / NSTAGE) - 1) & 1, P.err);
                if (!ok) break;
                const int nt = min(NCWARP, nT - s * NCWARP);
                const int tok = t0 + s * STAGE_TOK;
                const uint32_t kc_b = nt * 1024;
                const int ngrp = (nt * 32 + G - 1) / G;
                const uint32_t ksz_b = ngrp * KVQ_D * 4;
                const uint32_t vc_b = nt * 32 * (KVQ_D / 4);
                const uint32_t vsz_b = nt * 32 * (KVQ_D / Gv) * 4;
                uint8_t *st = S.stage[slot];
                mbar_expect_tx(&S.full[slot], kc_b + ksz_b + vc_b + vsz_b);
                bulk_g2s(st, kc_base + (int64_t)(tok >> 5) * 1024, kc_b, &S.full[slot]);
                bulk_g2s(st + KC_BYTES, ksz_base + (int64_t)(tok / G) * KVQ_D, ksz_b, &S.full[slot]);
                bulk_g2s(st + KC_BYTES + KSZ_MAX, vc_base + (int64_t)tok * (KVQ_D / 4), vc_b, &S.full[slot]);
                bulk_g2s(st + KC_BYTES + KSZ_MAX + VC_BYTES, vsz_base + (int64_t)tok * (KVQ_D / Gv), vsz_b,
                         &S.full[slot]);
            }
            // drain: every issued stage must have landed before the CTA exits
            const int issued = nstages;
            for (int s = max(0, issued - NSTAGE); s < issued; ++s) mbar_wait(&S.full[s % NSTAGE], (s / NSTAGE) & 1, P.err);
        }
        return;
    }

    // ---------------- consumers ----------------
    const uint16_t *qrow = P.q + ((int64_t)b * P.Hq + hq) * KVQ_D;
    float qa[4];
    {
        uint2 u = *reinterpret_cast<const uint2 *>(qrow + 4 * lane);
        qa[0] = h2f(lo16(u.x)) * P.alpha;
        qa[1] = h2f(hi16(u.x)) * P.alpha;
        qa[2] = h2f(lo16(u.y)) * P.alpha;
        qa[3] = h2f(hi16(u.y)) * P.alpha;
    }
    const int tq = lane & 3;                       // key mapping: lane = 4*(token quad) + channel block
    const int ts = lane >> 2, jg = lane & 3;       // value mapping: token slot, channel block of 32

    float m_run = -INFINITY, l_part = 0.f, vbias = 0.f;
    float vacc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) vacc[i] = 0.f;

    bool ok = true;
    for (int s = 0; s < nstages; ++s) {
        const int slot = s % NSTAGE;
        ok = ok && mbar_wait(&S.full[slot], (s / NSTAGE) & 1, P.err);
        const int tile = s * NCWARP + warp;
        if (ok && tile < nT) {
            const uint8_t *st = S.stage[slot];
            const int gl = (32 * warp) / G;                       // key group of this tile within the stage
            const uint32_t *ksz = reinterpret_cast<const uint32_t *>(st + KC_BYTES) + gl * KVQ_D;
            // ---- pre-scaled alpha*q*s of this group (fp32) and alpha*sum q z ----
            const float4 szv = *reinterpret_cast<const float4 *>(ksz + 4 * lane);
            const uint32_t sz0 = __float_as_uint(szv.x), sz1 = __float_as_uint(szv.y);
            const uint32_t sz2 = __float_as_uint(szv.z), sz3 = __float_as_uint(szv.w);
            // channel 4*lane + i has byte parity i & 1: pre-scale 2^(149-E0) or 2^(141-E0)
            const float pe = __int_as_float((127 + 149 - P.e0) << 23), po = __int_as_float((127 + 141 - P.e0) << 23);
            *reinterpret_cast<float4 *>(&S.qk[warp][4 * lane]) =
                make_float4(qa[0] * h2f(lo16(sz0)) * pe, qa[1] * h2f(lo16(sz1)) * po, qa[2] * h2f(lo16(sz2)) * pe,
                            qa[3] * h2f(lo16(sz3)) * po);
            const float cb = warp_sum(qa[0] * h2f(hi16(sz0)) + qa[1] * h2f(hi16(sz1)) + qa[2] * h2f(hi16(sz2)) +
                                      qa[3] * h2f(hi16(sz3)));
            __syncwarp();
            float qk[32];
            {
                const float4 *qs = reinterpret_cast<const float4 *>(&S.qk[warp][32 * tq]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 u = qs[i];
                    qk[4 * i] = u.x; qk[4 * i + 1] = u.y; qk[4 * i + 2] = u.z; qk[4 * i + 3] = u.w;
                }
            }
            // ---- key codes: tokens 4qd..4qd+3 x channels 32tq..32tq+31 ----
            const uint8_t *kt = st + warp * 1024;
            const uint4 ka = *reinterpret_cast<const uint4 *>(kt + lane * 16);
            const uint4 kb = *reinterpret_cast<const uint4 *>(kt + 512 + lane * 16);
            const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
            unsigned long long acc2[4] = {0ull, 0ull, 0ull, 0ull};     // fp32 pairs (0.0f, 0.0f)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t w0 = kw[k], w16 = kw[k] >> 16;          // bytes 0,1 | bytes 2,3 at bits 0..15
                const unsigned long long q01 = pack2f(qk[4 * k], qk[4 * k + 1]);
                const unsigned long long q23 = pack2f(qk[4 * k + 2], qk[4 * k + 3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t m0 = 3u << (2 * j), m1 = 3u << (8 + 2 * j);
                    acc2[j] = ffma2(pack2u(w0 & m0, w0 & m1), q01, acc2[j]);     // channels 4k, 4k+1
                    acc2[j] = ffma2(pack2u(w16 & m0, w16 & m1), q23, acc2[j]);   // channels 4k+2, 4k+3
                }
            }
            float acc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = lo2f(acc2[j]) + hi2f(acc2[j]);
            // transpose-reduce over the 4 lanes of the quad: lane keeps token 4qd + tq
            float score;
            {
                const bool h2 = (tq & 2) != 0;
                float s0 = h2 ? acc[0] : acc[2], s1 = h2 ? acc[1] : acc[3];
                float k0 = h2 ? acc[2] : acc[0], k1 = h2 ? acc[3] : acc[1];
                k0 += __shfl_xor_sync(0xFFFFFFFFu, s0, 2);
                k1 += __shfl_xor_sync(0xFFFFFFFFu, s1, 2);
                const bool h1 = (tq & 1) != 0;
                float sx = h1 ? k0 : k1;
                score = (h1 ? k1 : k0) + __shfl_xor_sync(0xFFFFFFFFu, sx, 1);
            }
            // undo the 2^(2j-E0) product scaling (j = tq), add the zero-point term
            const float logit = score * __int_as_float((127 + P.e0 - 2 * tq) << 23) + cb;
            // ---- online softmax over the tile (warp-uniform running max) ----
            const float mt = warp_max(logit);
            if (mt > m_run) {
                const float sc = exp2f(m_run - mt);
                l_part *= sc;
                vbias *= sc;
#pragma unroll
                for (int i = 0; i < 32; ++i) vacc[i] *= sc;
                m_run = mt;
            }
            const float p = exp2f(logit - m_run);
            l_part += p;
            // ---- values: 4 passes of 8 tokens; lane = (token slot ts, channel block jg) ----
            const uint8_t *vc = st + KC_BYTES + KSZ_MAX + warp * 32 * (KVQ_D / 4);
            const uint32_t *vsz = reinterpret_cast<const uint32_t *>(st + KC_BYTES + KSZ_MAX + VC_BYTES) +
                                  warp * 32 * (KVQ_D / Gv);
            const int jv = (32 * jg) / Gv;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int tau = 8 * r + ts;
                const float pt = __shfl_sync(0xFFFFFFFFu, p, tau);
                const uint32_t szt = vsz[tau * (KVQ_D / Gv) + jv];
                const uint16_t pp = f2h_rn(pt * h2f(lo16(szt)));
                vbias += pt * h2f(hi16(szt));
                const uint2 u = *reinterpret_cast<const uint2 *>(vc + tau * (KVQ_D / 4) + jg * 8);
                const uint32_t uw[2] = {u.x, u.y};
#pragma unroll
                for (int wi = 0; wi < 2; ++wi) {
                    const uint32_t w0 = uw[wi], w8 = uw[wi] >> 8;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t m = 0x00030003u << (2 * i);
                        const uint32_t e = w0 & m, o = w8 & m;
                        // channel 32jg + 16wi + 4b + i  ->  vacc[16wi + 4b + i]
                        vacc[16 * wi + 0 + i] = fma_f16f32(lo16(e), pp, vacc[16 * wi + 0 + i]);
                        vacc[16 * wi + 8 + i] = fma_f16f32(hi16(e), pp, vacc[16 * wi + 8 + i]);
                        vacc[16 * wi + 4 + i] = fma_f16f32(lo16(o), pp, vacc[16 * wi + 4 + i]);
                        vacc[16 * wi + 12 + i] = fma_f16f32(hi16(o), pp, vacc[16 * wi + 12 + i]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
    }

    // ---- fast-path state -> shared memory (channel order) ----
    {
        const float l_w = warp_sum(l_part);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float v = vacc[i];
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
            v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
            vacc[i] = v;
        }
        float vb = vbias;
        vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 4);
        vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 8);
        vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 16);
        // lane (ts, jg) writes channels 32jg + 4ts + i, i = 0..3 (idx = 16wi + 4b + i);
        // compile-time indices keep vacc in registers
#pragma unroll
        for (int idx = 0; idx < 32; ++idx)
            if ((idx >> 2) == ts)
                S.st_acc[2 * warp][32 * jg + idx] = vacc[idx] * __int_as_float((127 + 24 - 2 * (idx & 3)) << 23) + vb;
        if (lane == 0) {
            S.st_m[2 * warp] = m_run;
            S.st_l[2 * warp] = l_w;
        }
    }

    // ---- per-token path: tokens [max(t0, Qf), t1) (fp16 residual and partial tiles) ----
    {
        float m_g = -INFINITY, l_g = 0.f, ag[4] = {0.f, 0.f, 0.f, 0.f};
        const int gstart = max(t0, fast_end);
        const uint16_t *kres = P.k_res + bk * (int64_t)R * KVQ_D;
        const uint16_t *vres = P.v_res + bk * (int64_t)R * KVQ_D;
        for (int t = gstart + warp; t < t1; t += NCWARP) {
            float kv[4], vv[4];
            if (t < nKq) {
                const int gi = t / G, tt = t % G;
                const uint8_t *grp = kc_base + (int64_t)gi * ((int64_t)G * KVQ_D / 4);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = 4 * lane + i;
                    const int code = (grp[kivi_key_byte_offset(tt, c)] >> (2 * (tt & 3))) & 3;
                    const uint32_t szc = ksz_base[(int64_t)gi * KVQ_D + c];
                    kv[i] = (float)code * h2f(lo16(szc)) + h2f(hi16(szc));
                }
            } else {
                uint2 u = *reinterpret_cast<const uint2 *>(kres + (int64_t)(t % R) * KVQ_D + 4 * lane);
                kv[0] = h2f(lo16(u.x)); kv[1] = h2f(hi16(u.x)); kv[2] = h2f(lo16(u.y)); kv[3] = h2f(hi16(u.y));
            }
            if (t < nVq) {
                const uint8_t byte = vc_base[(int64_t)t * (KVQ_D / 4) + lane];
                const uint32_t szt = vsz_base[(int64_t)t * (KVQ_D / Gv) + (4 * lane) / Gv];
#pragma unroll
                for (int i = 0; i < 4; ++i) vv[i] = (float)((byte >> (2 * i)) & 3) * h2f(lo16(szt)) + h2f(hi16(szt));
            } else {
                uint2 u = *reinterpret_cast<const uint2 *>(vres + (int64_t)(t % R) * KVQ_D + 4 * lane);
                vv[0] = h2f(lo16(u.x)); vv[1] = h2f(hi16(u.x)); vv[2] = h2f(lo16(u.y)); vv[3] = h2f(hi16(u.y));
            }
            const float logit = warp_sum(qa[0] * kv[0] + qa[1] * kv[1] + qa[2] * kv[2] + qa[3] * kv[3]);
            const float mn = fmaxf(m_g, logit);
            const float sc = exp2f(m_g - mn);
            const float p = exp2f(logit - mn);
            l_g = l_g * sc + p;
#pragma unroll
            for (int i = 0; i < 4; ++i) ag[i] = ag[i] * sc + p * vv[i];
            m_g = mn;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) S.st_acc[2 * warp + 1][4 * lane + i] = ag[i];
        if (lane == 0) {
            S.st_m[2 * warp + 1] = m_g;
            S.st_l[2 * warp + 1] = l_g;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");

    // ---- merge the eight warp states, write (o_s, lse_s) ----
    if (warp == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < NSTATE; ++i) M = fmaxf(M, S.st_m[i]);
        float l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
        if (M > -INFINITY) {
#pragma unroll
            for (int i = 0; i < NSTATE; ++i) {
                const float w = S.st_m[i] > -INFINITY ? exp2f(S.st_m[i] - M) : 0.f;
                l += w * S.st_l[i];
#pragma unroll
                for (int c = 0; c < 4; ++c) o[c] += w * S.st_acc[i][4 * lane + c];
            }
        }
        const int64_t row = ((int64_t)b * P.Hq + hq) * P.splits + split;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float4 ov = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
        *reinterpret_cast<float4 *>(P.ws_o + row * KVQ_D + 4 * lane) = ov;
        if (lane == 0) P.ws_lse[row] = l > 0.f ? M + log2f(l) : -INFINITY;
    }
}

cudaError_t launch_decode_kivi(const kvq_config *cfg, const kvq_kivi_cache *c, const void *q, const DecodePlan &p,
                               void *ws, cudaStream_t st) {
    Params P;
    P.seq_len = c->seq_len;
    P.k_codes = static_cast<const uint8_t *>(c->k_codes);
    P.k_sz = static_cast<const uint32_t *>(c->k_sz);
    P.v_codes = static_cast<const uint8_t *>(c->v_codes);
    P.v_sz = static_cast<const uint32_t *>(c->v_sz);
    P.k_res = static_cast<const uint16_t *>(c->k_res);
    P.v_res = static_cast<const uint16_t *>(c->v_res);
    P.q = static_cast<const uint16_t *>(q);
    P.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_o);
    P.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_lse);
    P.err = device_error_ptr();
    P.Hq = cfg->n_q_heads;
    P.Hkv = cfg->n_kv_heads;
    P.G = cfg->group_k;
    P.Gv = cfg->group_v;
    P.R = cfg->residual;
    P.cap = ((int64_t)c->max_seq_len + 127) / 128 * 128;
    P.splits = p.splits;
    P.chunk = p.chunk;
    P.kgrp_cap = P.cap / cfg->group_k;
    P.alpha = sm_scale_of(cfg) * 1.4426950408889634f;
    // |alpha q s| < alpha 2^32 (fp16 q and s): 2^(149-E0) alpha 2^32 < 2^127
    P.e0 = 54 + (int)ceilf(log2f(P.alpha));
    if (P.e0 < 22) P.e0 = 22;
    if (!P.err) return cudaErrorInvalidDevicePointer;
    const size_t smem = sizeof(Smem);
    static int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kivi_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_dev = dev;
    }
    dim3 grid(p.splits, cfg->n_q_heads, c->batch);
    kivi_decode_kernel<<<grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kvq
