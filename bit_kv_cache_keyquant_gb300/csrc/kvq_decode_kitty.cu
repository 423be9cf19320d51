// a7: Kitty split-KV decode attention, stage 1.
//
// The cache of one (batch row, kv head): fp16 sink tokens [0, S); key pages
// of G = 128 tokens (two 2-bit planes, boost index, per-channel s, z),
// value pages (2-bit per-token codes, per-token s, z); an fp16 key Q-buffer,
// value Q-buffer and value local window (Kitty, "Page Structure for Key
// Cache", "Page Structure for Value Cache", "Stage 1: Inserting New KV
// Vectors").  A key code is X = low | (high << 2), high taken from row
// idx[c] of the high plane when idx[c] < K and 0 otherwise (Algorithm 1);
// K^ = X s + z.
//
// Structure (same as the KIVI stage-1 kernel): a persistent grid over
// (batch row, query head, split) units; a producer warp streams one page
// (key record + value record, 9856 B at K = 16) per stage with
// cp.async.bulk into a 4-slot mbarrier ring; four consumer warps each take
// 32 tokens of the page.  The low plane is stored in the KIVI key-tile order,
// so lane 4q + r finds its 32 channels (16k + 2r + {0, 1, 8, 9}) x 4 tokens
// (q + 8p) in two 16-byte chunks, and one word per 16 boosted rows (rows
// 16kh + 4r + {0..3}, weights 4 q s) in the high plane; the dot is the exact
// fp32 denormal-code x fma.rn.f32x2 form.  Values use the exact fp32
// token-major path (value_token_accum) with one (s, z) per token.
// The last split of every row covers every token outside whole pages of
// both sides (sink, buffers, local window, a key page whose values are
// still in fp16): one token per lane for the keys (per-lane independent
// loads), four channels per lane for the values.
#include "kvq_kitty.cuh"

namespace kvq {

namespace {

constexpr int NSTAGE = 4;
constexpr int QK_ROW = 36;

struct Smem {
    uint8_t stage[NSTAGE][STAGE_BYTES];
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    float qk[NCWARP][4 * QK_ROW];         // per-warp pre-scaled alpha q s (low plane)
    float hw[NCWARP][KMAX + 4];           // per-warp pre-scaled 4 alpha q s of the boosted rows
    float qv[KVQ_D];                       // alpha q (residual unit)
    float st_acc[NCWARP][KVQ_D];
    float st_m[NCWARP];
    float st_l[NCWARP];
    int abort_flag;                       // raised by a consumer warp whose wait gave up (last: the
                                          // members before it keep their 16-byte alignment)
};
static_assert(offsetof(Smem, qk) % 16 == 0 && offsetof(Smem, st_acc) % 16 == 0, "16-byte aligned tables");

__device__ __forceinline__ float softmax_tile(float logit, float &m_run, float &l_part, float &vbias,
                                              unsigned long long vacc2[16]) {
    const float mt = warp_max(logit);
    if (mt > m_run) {
        const float sc = exp2f(m_run - mt);
        l_part *= sc;
        vbias *= sc;
        scale_pairs(vacc2, sc);
        m_run = mt;
    }
    const float p = exp2f(logit - m_run);
    l_part += p;
    return p;
}

}  // namespace

__global__ void __launch_bounds__(32 * (NCWARP + 1), 4) kitty_decode_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_units = P.B * P.Hq * P.splits;
    const int K = P.K;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], NCWARP);
        }
        S.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCWARP) {
        if (lane == 0) kitty_produce<NSTAGE>(P, P.Hq, S.stage, S.full, S.empty, &S.abort_flag);
        return;
    }

    const int tq = lane & 3, qd = lane >> 2;
    const int ts = lane >> 2, jg = lane & 3;
    const float pe = __int_as_float((127 + 149 - P.e0) << 23), po = __int_as_float((127 + 141 - P.e0) << 23);
    const float lscale = __int_as_float((127 + P.e0 - 2 * tq) << 23);
    const int n_hgrp = (K + 15) / 16;          // groups of 16 boosted rows (4 per channel-block lane)
    bool ok = true;
    int sg = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = unit_of(P, u, P.Hq);
        float qa[4];
        {
            const uint2 qv = *reinterpret_cast<const uint2 *>(P.q + ((int64_t)U.b * P.Hq + U.hq) * KVQ_D + 4 * lane);
            qa[0] = h2f(lo16(qv.x)) * P.alpha;
            qa[1] = h2f(hi16(qv.x)) * P.alpha;
            qa[2] = h2f(lo16(qv.y)) * P.alpha;
            qa[3] = h2f(hi16(qv.y)) * P.alpha;
        }
        if (U.residual) {
            // ---------------- tokens outside whole pages ----------------
            if (warp == 0) *reinterpret_cast<float4 *>(&S.qv[4 * lane]) = make_float4(qa[0], qa[1], qa[2], qa[3]);
            asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
            float m_run, l_part, racc[4];
            kitty_residual(P, U, S.qv, warp, lane, racc, m_run, l_part);
            const float l_w = warp_sum(l_part);
            *reinterpret_cast<float4 *>(&S.st_acc[warp][4 * lane]) = make_float4(racc[0], racc[1], racc[2], racc[3]);
            if (lane == 0) {
                S.st_m[warp] = m_run;
                S.st_l[warp] = l_w;
            }
        } else {
            // lane = 8r + k writes the weights of channels c0 + {0, 1, 8, 9} = 16k + 2r + {0, 1, 8, 9}
            // (row r, word k of the table), pre-scaled by the byte-parity power of two
            const int c0 = 16 * (lane & 7) + 2 * (lane >> 3);
            float qf[4];
            {
                const uint16_t *qrow = P.q + ((int64_t)U.b * P.Hq + U.hq) * KVQ_D;
                const uint32_t q01 = *reinterpret_cast<const uint32_t *>(qrow + c0);
                const uint32_t q89 = *reinterpret_cast<const uint32_t *>(qrow + c0 + 8);
                qf[0] = h2f(lo16(q01)) * P.alpha;
                qf[1] = h2f(hi16(q01)) * P.alpha;
                qf[2] = h2f(lo16(q89)) * P.alpha;
                qf[3] = h2f(hi16(q89)) * P.alpha;
            }
            const float qp[4] = {qf[0] * pe, qf[1] * po, qf[2] * pe, qf[3] * po};
            float m_run = -INFINITY, l_part = 0.f, vbias = 0.f;
            unsigned long long vacc2[16];
#pragma unroll
for (int i = 0; i < 16; ++i) vacc2[i] = 0ull;
            for (int s = 0; s < U.np; ++s, ++sg) {
                const int slot = sg % NSTAGE;
                ok = consumer_stage_wait(&S.full[slot], (sg / NSTAGE) & 1, P.err, KVQ_SPIN_LIMIT, ok, &S.abort_flag);
                if (ok) {
                    const uint8_t *st = S.stage[slot];
                    const uint8_t *low = st, *high = st + KVQ_D * PG / 4, *idx = high + kitty_high_rows(K) * PG / 4;
                    const uint16_t *ps = reinterpret_cast<const uint16_t *>(idx + KVQ_D);
                    // ---- pre-scaled weights of the page: low plane (table order) and boosted rows ----
                    {
                        const uint32_t s01 = *reinterpret_cast<const uint32_t *>(ps + c0);
                        const uint32_t s89 = *reinterpret_cast<const uint32_t *>(ps + c0 + 8);
                        const float sv[4] = {h2f(lo16(s01)), h2f(hi16(s01)), h2f(lo16(s89)), h2f(hi16(s89))};
                        *reinterpret_cast<float4 *>(&S.qk[warp][(lane >> 3) * QK_ROW + 4 * (lane & 7)]) =
                            make_float4(qp[0] * sv[0], qp[1] * sv[1], qp[2] * sv[2], qp[3] * sv[3]);
                        const uint32_t i01 = *reinterpret_cast<const uint16_t *>(idx + c0);
                        const uint32_t i89 = *reinterpret_cast<const uint16_t *>(idx + c0 + 8);
                        const uint32_t id4 = i01 | (i89 << 16);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = (id4 >> (8 * i)) & 0xFF;
                            // boosted row r sits at byte r & 3 of its word: parity r & 1
                            if (r < K) S.hw[warp][r] = 4.f * qf[i] * sv[i] * ((r & 1) ? po : pe);
                        }
                        for (int r = K + lane; r < n_hgrp * 16; r += 32) S.hw[warp][r] = 0.f;   // rows past K
                    }
                    const uint32_t z01 = *reinterpret_cast<const uint32_t *>(ps + KVQ_D + c0);
                    const uint32_t z89 = *reinterpret_cast<const uint32_t *>(ps + KVQ_D + c0 + 8);
                    const float cb = warp_sum(qf[0] * h2f(lo16(z01)) + qf[1] * h2f(hi16(z01)) + qf[2] * h2f(lo16(z89)) +
                                              qf[3] * h2f(hi16(z89)));
                    __syncwarp();
                    // ---- key dot: tokens q + 8j (q = lane / 4), channels 16k + 2tq + {0, 1, 8, 9} ----
                    uint32_t kw[8];
                    {
                        const uint8_t *kt = low + warp * 1024;
                        const uint4 ka = *reinterpret_cast<const uint4 *>(kt + lane * 16);
                        const uint4 kb = *reinterpret_cast<const uint4 *>(kt + 512 + lane * 16);
                        kw[0] = ka.x; kw[1] = ka.y; kw[2] = ka.z; kw[3] = ka.w;
                        kw[4] = kb.x; kw[5] = kb.y; kw[6] = kb.z; kw[7] = kb.w;
                    }
                    const float4 *qs = reinterpret_cast<const float4 *>(&S.qk[warp][tq * QK_ROW]);
                    unsigned long long acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t w = kw[k];
                        const float4 qv = qs[k];
                        const uint32_t w16 = w >> 16;
                        const unsigned long long q01 = pack2f(qv.x, qv.y), q23 = pack2f(qv.z, qv.w);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t m0 = 3u << (2 * j), m1 = 3u << (8 + 2 * j);
                            acc2[j] = ffma2(pack2u(w & m0, w & m1), q01, acc2[j]);
                            acc2[j] = ffma2(pack2u(w16 & m0, w16 & m1), q23, acc2[j]);
                        }
                    }
                    // boosted rows 16hg + 4tq + b (b = 0..3) of this warp's tile block: weights 4 alpha q s,
                    // zero past K (a word past the plane's rows holds finite bytes of the stage)
                    const uint8_t *hb = high + warp * 8 * kitty_high_rows(K) + tq * 32 + qd * 4;
                    for (int hg = 0; hg < n_hgrp; ++hg) {
                        const int r0 = 16 * hg + 4 * tq;
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(hb + hg * 128);
                        const uint32_t w16 = w >> 16;
                        const unsigned long long q01 = pack2f(S.hw[warp][r0], S.hw[warp][r0 + 1]);
                        const unsigned long long q23 = pack2f(S.hw[warp][r0 + 2], S.hw[warp][r0 + 3]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t m0 = 3u << (2 * j), m1 = 3u << (8 + 2 * j);
                            acc2[j] = ffma2(pack2u(w & m0, w & m1), q01, acc2[j]);
                            acc2[j] = ffma2(pack2u(w16 & m0, w16 & m1), q23, acc2[j]);
                        }
                    }
                    float score;
                    {
                        const float a0 = lo2f(acc2[0]) + hi2f(acc2[0]), a1 = lo2f(acc2[1]) + hi2f(acc2[1]);
                        const float a2 = lo2f(acc2[2]) + hi2f(acc2[2]), a3 = lo2f(acc2[3]) + hi2f(acc2[3]);
                        const bool h2 = (tq & 2) != 0;
                        float k0 = h2 ? a2 : a0, k1 = h2 ? a3 : a1;
                        k0 += __shfl_xor_sync(0xFFFFFFFFu, h2 ? a0 : a2, 2);
                        k1 += __shfl_xor_sync(0xFFFFFFFFu, h2 ? a1 : a3, 2);
                        const bool h1 = (tq & 1) != 0;
                        score = (h1 ? k1 : k0) + __shfl_xor_sync(0xFFFFFFFFu, h1 ? k0 : k1, 1);
                    }
                    const float logit = score * lscale + cb;
                    const float p = softmax_tile(logit, m_run, l_part, vbias, vacc2);
                    // ---- values (token-major page, one (s, z) per token) ----
                    const uint8_t *vrec = st + VREC_OFF;
                    const uint8_t *vc = vrec + warp * 32 * (KVQ_D / 4);
                    const uint16_t *vs = reinterpret_cast<const uint16_t *>(vrec + PG * KVQ_D / 4) + 32 * warp;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int tau = 8 * r + ts;
                        const float pt = __shfl_sync(0xFFFFFFFFu, p, 4 * ts + r);   // lane 4q + tq holds token q + 8tq
                        vbias += pt * h2f(vs[PG + tau]);
                        value_token_accum(*reinterpret_cast<const uint2 *>(vc + tau * (KVQ_D / 4) + jg * 8), pt * h2f(vs[tau]), vacc2);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            // ---- warp state -> shared memory ----
            const float l_w = warp_sum(l_part);
            float vb = vbias;
            vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 4);
            vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 8);
            vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 16);
            float4 w4 = value_block_reduce<2>(vacc2, ts);
            w4.x += vb; w4.y += vb; w4.z += vb; w4.w += vb;
            *reinterpret_cast<float4 *>(&S.st_acc[warp][32 * jg + 4 * ts]) = w4;
            if (lane == 0) {
                S.st_m[warp] = m_run;
                S.st_l[warp] = l_w;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
        if (warp == 0) {
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < NCWARP; ++i) M = fmaxf(M, S.st_m[i]);
            float l = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M > -INFINITY) {
#pragma unroll
                for (int i = 0; i < NCWARP; ++i) {
                    const float w = S.st_m[i] > -INFINITY ? exp2f(S.st_m[i] - M) : 0.f;
                    l += w * S.st_l[i];
                    const float4 a = *reinterpret_cast<const float4 *>(&S.st_acc[i][4 * lane]);
                    o.x += w * a.x; o.y += w * a.y; o.z += w * a.z; o.w += w * a.w;
                }
            }
            const int64_t row = ((int64_t)U.b * P.Hq + U.hq) * P.splits + U.split;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            *reinterpret_cast<float4 *>(P.ws_o + row * KVQ_D + 4 * lane) =
                make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            if (lane == 0) P.ws_lse[row] = l > 0.f ? M + log2f(l) : -INFINITY;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
    }
}

cudaError_t launch_decode_kitty(const kvq_config *cfg, const kvq_kitty_cache *c, const void *q, const DecodePlan &p,
                                void *ws, cudaStream_t st) {
    Params P;
    P.seq_len = c->seq_len;
    P.k_pages = static_cast<const uint8_t *>(c->k_pages);
    P.v_pages = static_cast<const uint8_t *>(c->v_pages);
    P.page_table = c->page_table;
    P.n_pages = c->n_pages;
    P.k_sink = static_cast<const uint16_t *>(c->k_sink);
    P.v_sink = static_cast<const uint16_t *>(c->v_sink);
    P.k_qbuf = static_cast<const uint16_t *>(c->k_qbuf);
    P.v_qbuf = static_cast<const uint16_t *>(c->v_qbuf);
    P.v_local = static_cast<const uint16_t *>(c->v_local);
    P.q = static_cast<const uint16_t *>(q);
    P.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_o);
    P.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_lse);
    P.err = device_error_ptr();
    P.B = c->batch;
    P.Hq = cfg->n_q_heads;
    P.Hkv = cfg->n_kv_heads;
    P.S = cfg->sink;
    P.R = cfg->residual;
    P.K = cfg->boost_k;
    P.splits = p.splits;
    P.chunk = p.chunk;
    P.page_cap = (int)((c->max_seq_len - cfg->sink > 0 ? c->max_seq_len - cfg->sink : 0) + PG - 1) / PG;
    if (P.page_cap < 1) P.page_cap = 1;
    P.max_len = c->max_seq_len;
    P.vsub = 1;
    P.gall = cfg->n_q_heads / cfg->n_kv_heads;
    P.gu = P.gall;
    P.kpb = (int)kitty_key_page_bytes(cfg->boost_k);
    P.vpb = PG * KVQ_D / 4 + 4 * PG;
    P.alpha = sm_scale_of(cfg) * 1.4426950408889634f;
    P.e0 = 54 + (int)ceilf(log2f(P.alpha));
    if (P.e0 < 22) P.e0 = 22;
    if (!P.err) return cudaErrorInvalidDevicePointer;
    if (P.kpb > VREC_OFF || P.K > KMAX) return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(kitty_decode_kernel, smem, attr_done)) return e;
    const int64_t n_units = (int64_t)c->batch * cfg->n_q_heads * p.splits;
    int64_t grid = (int64_t)num_sms() * 4;
    if (grid > n_units) grid = n_units;
    kitty_decode_kernel<<<(unsigned)grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kvq
