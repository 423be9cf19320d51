// a7 for grouped-query heads: Kitty split-KV decode attention, stage 1, with
// all g <= 4 query heads of a kv head in one unit and both contractions on
// the tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulation).
//
// A page (Kitty, "Page-Centric Memory Layout and Dense-Sparse
// Decomposition") holds the key low plane, the high plane of the K boosted
// channels, the boost index and a per-channel (s, z); the value page holds
// token-major codes and a per-token (s, z).  The key code is X = low + 4 high,
// so
//   logit_ht = sum_c low_tc W_hc + sum_{r<K} high_tr 4 W_h,c(r) + alpha sum_c q_hc z_c
// with W_hc = alpha q_hc s_c: the dense low plane is eight 16-channel
// k-steps, the sparse high plane ceil(K/16) more k-steps whose B rows are
// the boosted channels' weights (dense-sparse decomposition on the tensor
// cores).  Both planes are stored in fragment order: the low plane as the
// KIVI 2-bit key tiles (lane 4q + r finds tokens q + 8p x channels
// 16k + 2r + {0, 1, 8, 9} of all eight k-steps in two 16-byte chunks), the
// high plane as one word per lane and 16-row k-step (rows 16kh + 4r + b at
// byte b; MMA k index 2r + e + 8h is row 4r + e + 2h).  Codes become exact
// fp16 operands through e4m3 bit patterns, weights are fp16 hi / lo pairs
// (see kvq_mma.cuh), with 2^sigma_h |alpha q| < 1/4 so that 4 W stays in
// fp16 range.  The B operands and the zero-point dot depend on the page, not
// on the tile: the four warps of a page build them once between them (warp
// w the low k-steps 2w, 2w + 1 and the high k-steps w, w + 4, ...) into a
// double-buffered shared copy, behind one barrier per page.
// Values are the per-token 2-bit codes of the KIVI grouped-query kernel with
// one (s, z) per token.  Tokens outside whole pages are the residual unit,
// per head on CUDA cores.
#include "kvq_kitty.cuh"
#include "kvq_mma.cuh"

namespace kvq {

namespace {

constexpr int KQ_NSTAGE = 3;
constexpr int KG_MAX = 4;                 // query heads per unit
constexpr int KPB_ROW = 40;               // p exchange row (32 tokens + 8): conflict-free stores
constexpr int KHK_MAX = (KMAX + 15) / 16;  // high-plane k-steps
constexpr int KACC_ROW = KVQ_D + 8;

struct SmemKG {
    uint8_t stage[KQ_NSTAGE][STAGE_BYTES];
    uint64_t full[KQ_NSTAGE];
    uint64_t empty[KQ_NSTAGE];
    uint32_t qhi[KG_MAX][64];             // fp16x2 hi parts of alpha q 2^sigma: [head][k/2][r][4]
    uint32_t qlo[KG_MAX][64];
    uint32_t qhl[KG_MAX][KVQ_D];          // channel order: fp16 hi | lo << 16 (the boosted rows' lookups)
    float qv[KVQ_D];                      // alpha q of one head, channel order (residual unit)
    float unsig[KG_MAX];                  // 2^-sigma_h
    uint8_t hchan[NCWARP][KMAX + 16];     // channel of boosted row r (per warp copy)
    float pbuf[NCWARP][KG_MAX * KPB_ROW];
    union {
        float st_acc[NCWARP][KG_MAX][KACC_ROW];   // warp states at the end of a unit
        struct {                                  // per page (double-buffered by stage parity)
            uint4 bk[2][4][32];                   // B words of low k-steps 2i, 2i+1: [buf][i][lane]
            uint2 bh[2][KHK_MAX][32];             // B words of high k-step hk: [buf][hk][lane]
            float zp[2][KG_MAX][NCWARP];          // zero-point dot of head h over k-steps 2w, 2w+1: [buf][h][w]
        } pg;
    };
    float st_m[NCWARP][KG_MAX];
    float st_l[NCWARP][KG_MAX];
    int abort_flag;                       // raised by a consumer warp whose wait gave up (last: the
                                          // members before it keep their 16-byte alignment)
};
static_assert(offsetof(SmemKG, qhi) % 16 == 0 && offsetof(SmemKG, qlo) % 16 == 0 && offsetof(SmemKG, st_acc) % 16 == 0,
              "16-byte aligned tables");
static_assert(sizeof(((SmemKG *)0)->pg) <= sizeof(((SmemKG *)0)->st_acc), "the page area fits the warp states");

}  // namespace

__global__ void __launch_bounds__(32 * (NCWARP + 1), 4) kitty_decode_gqa_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SmemKG &S = *reinterpret_cast<SmemKG *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // query heads per kv head (P.gall) and per unit (P.gu), units per batch row and split (Hkv vsub):
    // kernel parameters, read where used (no registers held across the tile loop)
    const int n_units = P.B * P.Hkv * P.vsub * P.splits;
    const int K = P.K;
    const int n_hk = (K + 15) >> 4;               // high-plane k-steps

    if (threadIdx.x == 0) {
        for (int i = 0; i < KQ_NSTAGE; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], NCWARP);
        }
        S.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCWARP) {
        if (lane == 0) kitty_produce<KQ_NSTAGE, true>(P, P.Hkv * P.vsub, S.stage, S.full, S.empty, &S.abort_flag);
        return;
    }

    const int q = lane >> 2, r = lane & 3;
    const int hB = q >> 1;
    const bool xB = (q & 1) != 0;
    // value codes: row address of this lane in the transposing matrix loads (matrix lane / 8: tokens
    // 8 (m % 2) + lane % 8 of a k-step, bytes 16 (m / 2) .. + 15 of their rows)
    const int vrow = 8 * ((lane >> 3) & 1) + (lane & 7), vcol = 16 * (lane >> 4);
    const uint32_t *qown = xB ? S.qlo[hB] : S.qhi[hB];   // the part of B column n = q (zero-point products)
    bool ok = true;
    int sg = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = unit_of<true>(P, u, P.Hkv * P.vsub);
        // first query row of the unit (recomputed where used: fewer live registers in the tile loop)
        auto hrow0 = [&]() { return (int64_t)U.b * P.Hq + (int64_t)(U.kvh * P.gall + U.sub * P.gu); };
        // ---- per-unit query tables: warp w prepares head w ----
        {
            const int h = warp;
            const int c0 = 16 * (lane & 7) + 2 * (lane >> 3);
            float qv[4] = {0.f, 0.f, 0.f, 0.f};
            if (h < P.gu) {
                const uint16_t *qrow = P.q + (hrow0() + h) * KVQ_D;
                const uint32_t q01 = *reinterpret_cast<const uint32_t *>(qrow + c0);
                const uint32_t q89 = *reinterpret_cast<const uint32_t *>(qrow + c0 + 8);
                qv[0] = h2f(lo16(q01)) * P.alpha;
                qv[1] = h2f(hi16(q01)) * P.alpha;
                qv[2] = h2f(lo16(q89)) * P.alpha;
                qv[3] = h2f(hi16(q89)) * P.alpha;
            }
            const float m = warp_max(fmaxf(fmaxf(fabsf(qv[0]), fabsf(qv[1])), fmaxf(fabsf(qv[2]), fabsf(qv[3]))));
            // 2^sigma m in [1/8, 1/4): |4 W| = |4 alpha q s| 2^sigma stays below 65504
            int ex = (int)((__float_as_uint(m) >> 23) & 255u) - 127;
            int sigma = m > 0.f ? -ex - 3 : 0;
            sigma = max(-120, min(120, sigma));
            const float sc = __int_as_float((127 + sigma) << 23);
            uint16_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v = qv[j] * sc;
                hi[j] = f2h_rn(v);
                lo[j] = f2h_rn(v - h2f(hi[j]));
            }
            const int tr = lane >> 3, tk = lane & 7;
            const int pw = (tk >> 1) * 16 + tr * 4 + 2 * (tk & 1);
            *reinterpret_cast<uint2 *>(&S.qhi[h][pw]) =
                make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
            *reinterpret_cast<uint2 *>(&S.qlo[h][pw]) =
                make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
            S.qhl[h][c0] = (uint32_t)hi[0] | ((uint32_t)lo[0] << 16);
            S.qhl[h][c0 + 1] = (uint32_t)hi[1] | ((uint32_t)lo[1] << 16);
            S.qhl[h][c0 + 8] = (uint32_t)hi[2] | ((uint32_t)lo[2] << 16);
            S.qhl[h][c0 + 9] = (uint32_t)hi[3] | ((uint32_t)lo[3] << 16);
            if (lane == 0) S.unsig[h] = __int_as_float((127 - sigma) << 23);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");

        if (U.residual) {
            for (int h = 0; h < P.gu; ++h) {
                if (warp == 0) {
                    const uint16_t *qrow = P.q + (hrow0() + h) * KVQ_D;
                    const uint2 qr = *reinterpret_cast<const uint2 *>(qrow + 4 * lane);
                    *reinterpret_cast<float4 *>(&S.qv[4 * lane]) =
                        make_float4(h2f(lo16(qr.x)) * P.alpha, h2f(hi16(qr.x)) * P.alpha, h2f(lo16(qr.y)) * P.alpha,
                                    h2f(hi16(qr.y)) * P.alpha);
                }
                asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
                float m_run, l_part, racc[4];
                kitty_residual(P, U, S.qv, warp, lane, racc, m_run, l_part);
                const float l_w = warp_sum(l_part);
                *reinterpret_cast<float4 *>(&S.st_acc[warp][h][4 * lane]) = make_float4(racc[0], racc[1], racc[2], racc[3]);
                if (lane == 0) {
                    S.st_m[warp][h] = m_run;
                    S.st_l[warp][h] = l_w;
                }
                asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
            }
        } else {
            float m_run = -INFINITY, l_part = 0.f;   // head r
            float vzacc[4] = {0.f, 0.f, 0.f, 0.f};   // sum_t p z_t of head r (hi, lo; rows q, q + 8 alike)
            float vacc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) vacc[i][0] = vacc[i][1] = vacc[i][2] = vacc[i][3] = 0.f;
            const float unsig = S.unsig[r];
            for (int s = 0; s < U.np; ++s, ++sg) {
                const int slot = sg % KQ_NSTAGE;
                ok = consumer_stage_wait(&S.full[slot], (sg / KQ_NSTAGE) & 1, P.err, KVQ_SPIN_LIMIT, ok, &S.abort_flag);
                const int buf = sg & 1;
                const uint8_t *st = S.stage[slot];
                const uint8_t *low = st, *high = st + KVQ_D * PG / 4, *idx = high + kitty_high_rows(K) * PG / 4;
                const uint16_t *ks = reinterpret_cast<const uint16_t *>(idx + KVQ_D);   // s [D], then z [D]
                if (ok) {
                    // ---- this warp's share of the page's B operands (column n = q: head hB, part xB) ----
                    {
                        const int i = warp;                       // low k-steps 2i, 2i + 1
                        const uint4 a = *reinterpret_cast<const uint4 *>(&S.qhi[hB][16 * i + 4 * r]);
                        const uint4 l = *reinterpret_cast<const uint4 *>(&S.qlo[hB][16 * i + 4 * r]);
                        const uint4 qo = *reinterpret_cast<const uint4 *>(qown + 16 * i + 4 * r);
                        uint32_t sv[4];
                        float zd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const int c0 = 16 * (2 * i + kk) + 2 * r;
                            sv[2 * kk] = *reinterpret_cast<const uint32_t *>(ks + c0);
                            sv[2 * kk + 1] = *reinterpret_cast<const uint32_t *>(ks + c0 + 8);
                            // alpha sum_c q_hc z_c as a product: A = the page's z_c in every row, B = the lane's part
                            // of alpha q 2^sigma
                            const uint32_t z01 = *reinterpret_cast<const uint32_t *>(ks + KVQ_D + c0);
                            const uint32_t z89 = *reinterpret_cast<const uint32_t *>(ks + KVQ_D + c0 + 8);
                            mma16816(zd, z01, z01, z89, z89, kk ? qo.z : qo.x, kk ? qo.w : qo.y);
                        }
                        S.pg.bk[buf][i][lane] = make_uint4(split_prod(a.x, l.x, sv[0], xB), split_prod(a.y, l.y, sv[1], xB),
                                                           split_prod(a.z, l.z, sv[2], xB), split_prod(a.w, l.w, sv[3], xB));
                        if (q == 0) S.pg.zp[buf][r][warp] = zd[0] + zd[1];   // head r: hi + lo parts
                    }
                    if (warp < n_hk) {
                        // boosted-row channel table of this page
                        const uint32_t id4 = *reinterpret_cast<const uint32_t *>(idx + 4 * lane);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int rr = (id4 >> (8 * i)) & 0xFF;
                            if (rr < K) S.hchan[warp][rr] = (uint8_t)(4 * lane + i);
                        }
                        for (int rr = K + lane; rr < 16 * n_hk; rr += 32) S.hchan[warp][rr] = 0xFF;   // rows past K
                        __syncwarp();
                        for (int hk = warp; hk < n_hk; hk += NCWARP) {
                            // rows 16hk + 4r + {0, 1} (first register) and + {2, 3} (second): B = 4 W of their
                            // channels, 0 past K
                            const int r0 = 16 * hk + 4 * r;
                            uint32_t bw[2];
#pragma unroll
                            for (int jp = 0; jp < 2; ++jp) {
                                const int ca = S.hchan[warp][r0 + 2 * jp], cb = S.hchan[warp][r0 + 2 * jp + 1];
                                const uint32_t ha = ca < KVQ_D ? S.qhl[hB][ca] : 0u, hb = cb < KVQ_D ? S.qhl[hB][cb] : 0u;
                                const uint32_t sa = ca < KVQ_D ? (uint32_t)ks[ca] : 0u, sb = cb < KVQ_D ? (uint32_t)ks[cb] : 0u;
                                // 4 W = (4 qhi) s + ...: scaling the query parts by 4 is exact
                                bw[jp] = split_prod(hmul2(prmt(ha, hb, 0x5410u), 0x44004400u),
                                                    hmul2(prmt(ha, hb, 0x7632u), 0x44004400u), sa | (sb << 16), xB);
                            }
                            S.pg.bh[buf][hk][lane] = make_uint2(bw[0], bw[1]);
                        }
                    }
                }
                // every warp at every page, also one whose wait gave up: the page's B operands are complete
                asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
                if (ok) {
                    // ---- low plane x W, then the boosted rows x 4W, on the tensor cores ----
                    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
                    {
                        const uint8_t *kt = low + warp * 1024;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint2 kw = *reinterpret_cast<const uint2 *>(kt + 512 * (i >> 1) + lane * 16 + 8 * (i & 1));
                            const uint4 b = S.pg.bk[buf][i][lane];
                            const uint32_t bk[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t w = kk ? kw.y : kw.x, w4 = w >> 4;
                                uint32_t a0l, a0h, a1l, a1h, a2l, a2h, a3l, a3h;
                                e4m3x4_f16x2(w & 0x03030303u, a0l, a0h);
                                e4m3x4_f16x2(w & 0x0C0C0C0Cu, a1l, a1h);
                                e4m3x4_f16x2(w4 & 0x03030303u, a2l, a2h);
                                e4m3x4_f16x2(w4 & 0x0C0C0C0Cu, a3l, a3h);
                                mma16816(s0, a0l, a1l, a0h, a1h, bk[2 * kk], bk[2 * kk + 1]);
                                mma16816(s1, a2l, a3l, a2h, a3h, bk[2 * kk], bk[2 * kk + 1]);
                            }
                        }
                        // boosted rows: one word of this warp's tile block per 16-row k-step (a word past the
                        // plane's rows holds finite bytes of the stage; its B rows are zero)
                        const uint8_t *hw = high + warp * 8 * kitty_high_rows(K) + r * 32 + q * 4;
                        for (int hk = 0; hk < n_hk; ++hk) {
                            const uint32_t w = *reinterpret_cast<const uint32_t *>(hw + hk * 128), w4 = w >> 4;
                            const uint2 b = S.pg.bh[buf][hk][lane];
                            uint32_t a0l, a0h, a1l, a1h, a2l, a2h, a3l, a3h;
                            e4m3x4_f16x2(w & 0x03030303u, a0l, a0h);
                            e4m3x4_f16x2(w & 0x0C0C0C0Cu, a1l, a1h);
                            e4m3x4_f16x2(w4 & 0x03030303u, a2l, a2h);
                            e4m3x4_f16x2(w4 & 0x0C0C0C0Cu, a3l, a3h);
                            mma16816(s0, a0l, a1l, a0h, a1h, b.x, b.y);
                            mma16816(s1, a2l, a3l, a2h, a3h, b.x, b.y);
                        }
                    }
                    // ---- logits of head r, tokens q, q + 8, q + 16, q + 24; online softmax ----
                    const float f9 = unsig * 512.f, f7 = unsig * 128.f;
                    float zr;
                    {
                        const float4 zq = *reinterpret_cast<const float4 *>(S.pg.zp[buf][r]);
                        zr = ((zq.x + zq.y) + (zq.z + zq.w)) * unsig;
                    }
                    float lg[4];
                    lg[0] = fmaf(s0[0] + s0[1], f9, zr);
                    lg[1] = fmaf(s0[2] + s0[3], f7, zr);
                    lg[2] = fmaf(s1[0] + s1[1], f9, zr);
                    lg[3] = fmaf(s1[2] + s1[3], f7, zr);
                    float mt = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
                    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 4));
                    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 8));
                    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 16));
                    // rescale when a head of the warp raised its maximum: a warp-uniform branch (the heads'
                    // lanes would diverge), the other heads' lanes multiplying by 1
                    if (__any_sync(0xFFFFFFFFu, mt > m_run)) {
                        const float mn = fmaxf(m_run, mt);
                        const float sc = ex2_ftz(m_run - mn);
                        l_part *= sc;
                        scale4(vzacc, sc);
#pragma unroll
                        for (int i = 0; i < 8; ++i) scale4(vacc[i], sc);
                        m_run = mn;
                    }
                    float pr[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        pr[i] = ex2_ftz(lg[i] - m_run);
                        l_part += pr[i];
                    }
                    // p of head r, token q + 8i, at position q + 8i of row r
                    float *pb = S.pbuf[warp];
#pragma unroll
                    for (int i = 0; i < 4; ++i) pb[r * KPB_ROW + q + 8 * i] = pr[i];
                    const uint8_t *vrec = st + VREC_OFF;
                    const uint16_t *vs = reinterpret_cast<const uint16_t *>(vrec + PG * KVQ_D / 4) + 32 * warp;
                    __syncwarp();
                    // ---- values: k-column k of k-step kv is token 16kv + k; A from transposing matrix loads of
                    //      the token-major code rows: a lane's word holds bytes 2q, 2q + 1 of tokens 2r, 2r + 1
                    //      (channels 8q .. 8q + 7 of a 64-channel half), m-tile 4hh + j takes channel 8q + j
                    //      (row q) and 8q + 4 + j (row q + 8) of half hh ----
                    const uint8_t *vc = vrec + warp * 32 * (KVQ_D / 4);
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        const float2 pa = *reinterpret_cast<const float2 *>(&pb[hB * KPB_ROW + 16 * kv + 2 * r]);
                        const float2 pc = *reinterpret_cast<const float2 *>(&pb[hB * KPB_ROW + 16 * kv + 8 + 2 * r]);
                        const uint32_t pha = split_pair(pa.x, pa.y, false), pla = split_pair(pa.x, pa.y, true);
                        const uint32_t phc = split_pair(pc.x, pc.y, false), plc = split_pair(pc.x, pc.y, true);
                        const uint32_t sa = *reinterpret_cast<const uint32_t *>(vs + 16 * kv + 2 * r);
                        const uint32_t sc8 = *reinterpret_cast<const uint32_t *>(vs + 16 * kv + 8 + 2 * r);
                        const uint32_t bv0 = split_prod(pha, pla, sa, xB);
                        const uint32_t bv1 = split_prod(phc, plc, sc8, xB);
                        {
                            // value zero-point product: A rows hold z of the k-step's tokens, B the lane's part of p
                            const uint32_t za = *reinterpret_cast<const uint32_t *>(vs + PG + 16 * kv + 2 * r);
                            const uint32_t zc = *reinterpret_cast<const uint32_t *>(vs + PG + 16 * kv + 8 + 2 * r);
                            mma16816(vzacc, za, za, zc, zc, xB ? pla : pha, xB ? plc : phc);
                        }
                        uint32_t m4[4];
                        ldsm_x4_trans(m4, vc + (16 * kv + vrow) * 32 + vcol);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            // tokens 2r, 2r + 1 (x) and 2r + 8, 2r + 9 (y): bytes 2q of both, then 2q + 1 of both
                            const uint32_t x = prmt(m4[2 * hh], 0u, 0x3120u), y = prmt(m4[2 * hh + 1], 0u, 0x3120u);
                            const uint32_t x4 = x >> 4, y4 = y >> 4;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t mk = (j & 1) ? 0x0C0C0C0Cu : 0x03030303u;
                                uint32_t a0, a1, a2, a3;
                                e4m3x4_f16x2((j < 2 ? x : x4) & mk, a0, a1);
                                e4m3x4_f16x2((j < 2 ? y : y4) & mk, a2, a3);
                                mma16816(vacc[4 * hh + j], a0, a1, a2, a3, bv0, bv1);
                            }
                        }
                    }
                    __syncwarp();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            // ---- warp state (head r) -> shared memory (over the page area: every warp is past its last page) ----
            asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
            float l_w = l_part;
            l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 4);
            l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 8);
            l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 16);
            const float vz = vzacc[0] + vzacc[1];
            float *acc = S.st_acc[warp][r];
            // m-tile 4hh + j: row q is channel 64hh + 8q + j, row q + 8 channel 64hh + 8q + 4 + j, codes
            // x 2^-9 (j even) or 2^-7 (j odd)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float (*v)[4] = &vacc[4 * hh];
                *reinterpret_cast<float4 *>(&acc[64 * hh + 8 * q]) =
                    make_float4(fmaf(v[0][0] + v[0][1], 512.f, vz), fmaf(v[1][0] + v[1][1], 128.f, vz),
                                fmaf(v[2][0] + v[2][1], 512.f, vz), fmaf(v[3][0] + v[3][1], 128.f, vz));
                *reinterpret_cast<float4 *>(&acc[64 * hh + 8 * q + 4]) =
                    make_float4(fmaf(v[0][2] + v[0][3], 512.f, vz), fmaf(v[1][2] + v[1][3], 128.f, vz),
                                fmaf(v[2][2] + v[2][3], 512.f, vz), fmaf(v[3][2] + v[3][3], 128.f, vz));
            }
            if (q == 0) {
                S.st_m[warp][r] = m_run;
                S.st_l[warp][r] = l_w;
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
        // ---- warp w merges head w over the four warp states, writes (o_s, lse_s) ----
        if (warp < P.gu) {
            const int h = warp;
            float M = -INFINITY;
#pragma unroll
            for (int i = 0; i < NCWARP; ++i) M = fmaxf(M, S.st_m[i][h]);
            float l = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M > -INFINITY) {
#pragma unroll
                for (int i = 0; i < NCWARP; ++i) {
                    const float w = S.st_m[i][h] > -INFINITY ? exp2f(S.st_m[i][h] - M) : 0.f;
                    l += w * S.st_l[i][h];
                    const float4 a = *reinterpret_cast<const float4 *>(&S.st_acc[i][h][4 * lane]);
                    o.x += w * a.x; o.y += w * a.y; o.z += w * a.z; o.w += w * a.w;
                }
            }
            const int64_t row = (hrow0() + h) * P.splits + U.split;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            *reinterpret_cast<float4 *>(P.ws_o + row * KVQ_D + 4 * lane) =
                make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
            if (lane == 0) P.ws_lse[row] = l > 0.f ? M + log2f(l) : -INFINITY;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
    }
}

// 2 <= g <= 4 heads per kv head in one unit, or an even g <= 8 in two units of g / 2 heads
int kitty_gqa_units_per_kv_head(const kvq_config *cfg) {
    const int g = cfg->n_q_heads / cfg->n_kv_heads;
    return g > KG_MAX ? 2 : 1;
}

bool kitty_gqa_supported(const kvq_config *cfg) {
    const int g = cfg->n_q_heads / cfg->n_kv_heads;
    return g >= 2 && (g <= KG_MAX || (g <= 2 * KG_MAX && g % 2 == 0));
}

cudaError_t launch_decode_kitty_gqa(const kvq_config *cfg, const kvq_kitty_cache *c, const void *q,
                                    const DecodePlan &p, void *ws, cudaStream_t st) {
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
    P.kpb = (int)kitty_key_page_bytes(cfg->boost_k);
    P.vpb = PG * KVQ_D / 4 + 4 * PG;
    P.alpha = sm_scale_of(cfg) * 1.4426950408889634f;
    P.e0 = 0;
    if (!P.err) return cudaErrorInvalidDevicePointer;
    if (P.kpb > VREC_OFF || P.K > KMAX) return cudaErrorInvalidValue;
    const size_t smem = sizeof(SmemKG);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(kitty_decode_gqa_kernel, smem, attr_done)) return e;
    P.vsub = kitty_gqa_units_per_kv_head(cfg);
    P.gall = cfg->n_q_heads / cfg->n_kv_heads;
    P.gu = P.gall / P.vsub;
    const int64_t n_units = (int64_t)c->batch * cfg->n_kv_heads * P.vsub * p.splits;
    int64_t grid = (int64_t)num_sms() * 4;
    if (grid > n_units) grid = n_units;
    kitty_decode_gqa_kernel<<<(unsigned)grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kvq
