// a3 for grouped-query heads: KIVI split-KV decode attention, stage 1, with
// all g <= 4 query heads of a kv head in one work unit and both contractions
// on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulation).
// Each packed code is unpacked once and serves every head of its kv head.
//
// Keys (KIVI Eq. 3 with the dequantization folded out):
//   S[t, n] = sum_c A[t, c] B[c, n]            n = 2h + x, x = 0 (hi), 1 (lo)
//   A[t, c] = code_tc * 2^-9 or 2^-7: the packed byte is masked into an e4m3
//             bit pattern (2-bit code in the low mantissa bits, or straddling
//             the mantissa and the exponent's low bit, both linear in the
//             code) and converted exactly with cvt.rn.f16x2.e4m3x2;
//   B[c, n] = fp16 hi / lo parts of W = alpha q_hc s_c 2^sigma_h.  With the
//             query split once per unit into fp16 qhi + qlo, hi = fl(qhi s)
//             and lo = fl(qlo s + (qhi s - hi)); the bracket is the exact
//             rounding error of hi (one fp16 FMA), so hi + lo carries W to
//             about 2^-21 relative, and sigma_h keeps every part in range.
//   logit_ht = (S[t, 2h] + S[t, 2h+1]) 2^(9|7 - sigma_h) + alpha sum_c q_hc z_c,
//   the zero-point term as one more product per k-step: A = the group's z_c
//   (fp16, exact) in every row, B = the hi / lo parts of alpha q_hc 2^sigma_h.
// Values:
//   O[c, n]  = sum_t A[c, t] B[t, n]
//   A[c, t] = code_tc * 2^-9 or 2^-7 (same unpacking, channel rows; the
//             cache's value tiles hold each lane's A words of a 16-token
//             k-step in one 16-byte chunk at 2 bits, two at 4 bits);
//   B[t, n] = hi / lo parts of p_ht s_tg (p kept as fp16 hi + lo);
//   o_hc     = (O[c, 2h] + O[c, 2h+1]) 2^(9|7) + sum_t p_ht z_tg,
//   the zero-point term again on the tensor cores: A row g = z_tg (rows
//   repeat the D/Gv groups), B = the hi / lo parts of p_ht.
// Products on the tensor cores are exact (fp16 x fp16) and accumulate in
// fp32; A operands are normal fp16 numbers (subnormal A operands lose bits).
//
// Work decomposition as the per-head kernel: a persistent grid walks the
// (batch row, kv head, split) units; a producer warp streams 128-token
// stages with bulk async copies into an mbarrier ring; four consumer warps
// each take one 32-token tile (two 16-token m-tiles) per stage; the last
// split of every row is the residual unit, done per head on CUDA cores.
// Three CTAs per SM with a three-stage ring: 12 consumer warps at 128
// registers, no spills (measured 3-6 % faster on the grouped-query layers
// than four CTAs at 96 registers, which spill in the tile loop).
#include "kvq_kivi.cuh"
#include "kvq_mma.cuh"

namespace kvq {

namespace {

constexpr int GMAX = 4;                   // query heads per unit (n = 8 tensor-core columns)
constexpr int PB_ROW = 40;                // p exchange row: 32 tokens + 8 floats (conflict-free)
constexpr int ACC_ROW = KVQ_D + 8;

template <int BK, int BV, int NST>
struct SmemG {
    uint8_t stage[NST][Geo<BK, BV>::BYTES];
    uint64_t full[NST];
    uint64_t empty[NST];
    uint32_t qhi[GMAX][64];               // fp16x2 hi parts of alpha q 2^sigma: [head][k/2][r][4]
    uint32_t qpad[16];                    // puts qlo's chunks on the other half of the banks
    uint32_t qlo[GMAX][64];               // fp16x2 lo parts, same order
    float qz[GMAX][KVQ_D];                // alpha q (fp32): [head][k][r][4] (4-bit widths' zero-point dots)
    float unsig[GMAX];                    // 2^-sigma_h
    float pbuf[NCWARP][GMAX * PB_ROW];
    float st_acc[NCWARP][GMAX][ACC_ROW];
    float st_m[NCWARP][GMAX];
    float st_l[NCWARP][GMAX];
    int abort_flag;                       // raised by a consumer warp whose wait gave up (last: the
                                          // members before it keep their 16-byte alignment)
};
// members read with 16-byte vector loads stay 16-byte aligned
using SmemG_223 = SmemG<2, 2, 3>;
using SmemG_442 = SmemG<4, 4, 2>;
static_assert(offsetof(SmemG_223, qhi) % 16 == 0 && offsetof(SmemG_223, qlo) % 16 == 0 &&
                  offsetof(SmemG_223, qz) % 16 == 0 && offsetof(SmemG_223, st_acc) % 16 == 0 &&
                  offsetof(SmemG_442, qhi) % 16 == 0 && offsetof(SmemG_442, st_acc) % 16 == 0,
              "16-byte aligned shared-memory tables");

}  // namespace

// BK-bit keys and BV-bit values (2 or 4) in an NST-stage ring.
template <int NGV, int BK, int BV, int NST>
__global__ void __launch_bounds__(32 * (NCWARP + 1), 3) kivi_decode_gqa_kernel(Params P) {
    using GG = Geo<BK, BV>;
    constexpr int GQ_NSTAGE = NST;
    // zero-point terms as tensor-core products (2-bit widths) or as CUDA-core dots (4-bit widths: the
    // products' extra registers cost the 4-bit variants more in spills than they save)
    constexpr bool ZMMA = BK == 2 && BV == 2;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SmemG<BK, BV, NST> &S = *reinterpret_cast<SmemG<BK, BV, NST> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // query heads per kv head (P.gall) and per unit (P.gu), units per batch row and split (Hkv vsub):
    // kernel parameters, read where used (no registers held across the tile loop)
    const int n_units = P.B * P.Hkv * P.vsub * P.splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < GQ_NSTAGE; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], NCWARP);
        }
        S.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCWARP) {
        if (lane == 0) kivi_produce<GQ_NSTAGE, true, BK, BV>(P, P.Hkv * P.vsub, S.stage, S.full, S.empty, &S.abort_flag);
        return;
    }

    // ---------------- consumers ----------------
    const int q = lane >> 2, r = lane & 3;         // mma group id / thread in group
    const int hB = q >> 1;                         // head of this lane's B column (n = q)
    const bool xB = (q & 1) != 0;                  // B column holds lo parts
    const int gl = (32 * warp) / P.G;              // key group of this warp's tile within a stage
    const uint32_t *qown = xB ? S.qlo[hB] : S.qhi[hB];   // the part of B column n = q (zero-point products)
    const int jz = q % NGV;                               // value group of rows q, q + 8 of the zero-point product
    bool ok = true;
    int sg = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = unit_of<true>(P, u, P.Hkv * P.vsub);
        // first query row of the unit (recomputed where used: fewer live registers in the tile loop)
        auto hrow0 = [&]() { return (int64_t)U.b * P.Hq + (int64_t)(U.kvh * P.gall + U.sub * P.gu); };
        // ---- per-unit query tables: warp w prepares head w ----
        {
            const int h = warp;
            const int c0 = 16 * (lane & 7) + 2 * (lane >> 3);   // entries 4*lane..4*lane+3
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
            // 2^sigma m in [1/2, 1): every |W| = |alpha q s| 2^sigma stays below 65504
            int ex = (int)((__float_as_uint(m) >> 23) & 255u) - 127;
            int sigma = m > 0.f ? -ex - 1 : 0;
            sigma = max(-120, min(120, sigma));
            const float sc = __int_as_float((127 + sigma) << 23);
            uint16_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v = qv[j] * sc;
                hi[j] = f2h_rn(v);
                lo[j] = f2h_rn(v - h2f(hi[j]));
            }
            // lane = 8r + k holds channels 16k + 2r + {0, 1, 8, 9}
            const int tr = lane >> 3, tk = lane & 7;
            const int pw = (tk >> 1) * 16 + tr * 4 + 2 * (tk & 1);
            *reinterpret_cast<uint2 *>(&S.qhi[h][pw]) =
                make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
            *reinterpret_cast<uint2 *>(&S.qlo[h][pw]) =
                make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
            if (!ZMMA) *reinterpret_cast<float4 *>(&S.qz[h][tk * 16 + tr * 4]) = make_float4(qv[0], qv[1], qv[2], qv[3]);
            if (lane == 0) S.unsig[h] = __int_as_float((127 - sigma) << 23);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");

        if (U.residual) {
            for (int h = 0; h < P.gu; ++h) {
                const uint16_t *qrow = P.q + (hrow0() + h) * KVQ_D;
                const uint2 qr = *reinterpret_cast<const uint2 *>(qrow + 4 * lane);
                const float qa[4] = {h2f(lo16(qr.x)) * P.alpha, h2f(hi16(qr.x)) * P.alpha, h2f(lo16(qr.y)) * P.alpha,
                                     h2f(hi16(qr.y)) * P.alpha};
                float m_run, l_part, racc[4];
                kivi_residual(P, U, qa, warp, lane, racc, m_run, l_part);
                const float l_w = warp_sum(l_part);
                *reinterpret_cast<float4 *>(&S.st_acc[warp][h][4 * lane]) = make_float4(racc[0], racc[1], racc[2], racc[3]);
                if (lane == 0) {
                    S.st_m[warp][h] = m_run;
                    S.st_l[warp][h] = l_w;
                }
            }
        } else {
            float m_run = -INFINITY, l_part = 0.f;        // head r
            float vzacc[4] = {0.f, 0.f, 0.f, 0.f};        // sum_t p z_t,jz of head r (hi, lo; rows q, q + 8)
            float vzc[NGV];                               // the CUDA-core form: sum_t p z_t,j of head r
#pragma unroll
            for (int i = 0; i < NGV; ++i) vzc[i] = 0.f;
            float vacc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) vacc[i][0] = vacc[i][1] = vacc[i][2] = vacc[i][3] = 0.f;
            const float unsig = S.unsig[r];
            for (int s = 0; s < U.nstages; ++s, ++sg) {
                const int slot = sg % GQ_NSTAGE;
                ok = consumer_stage_wait(&S.full[slot], (sg / GQ_NSTAGE) & 1, P.err, KIVI_WAIT_LIMIT(P), ok, &S.abort_flag);
                const int tile = s * NCWARP + warp;
                if (ok && tile < U.nT) {
                    const uint8_t *st = S.stage[slot];
                    const uint16_t *ksz = reinterpret_cast<const uint16_t *>(st + GG::KC) + gl * 2 * KVQ_D;
                    // ---- key codes x B on the tensor cores: tokens q + 8p, p = 0..3; B fragments (head hB,
                    //      hi or lo) of channels 16k + 2r + {0,1 | 8,9} made two k-steps at a time ----
                    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
                    float z0[4] = {0.f, 0.f, 0.f, 0.f}, z1[4] = {0.f, 0.f, 0.f, 0.f};   // two chains
                    {
                        // BK = 4: plane 0 holds tokens p = 0, 1, plane 1 tokens p = 2, 3, a nibble each
                        const uint8_t *kt = st + warp * 512 * BK;
                        // plane-0 key words: at 2 bits loaded per k-step pair where used, at 4 bits all up front
                        // (each measured faster for its width: register pressure differs)
                        uint4 ka = make_uint4(0u, 0u, 0u, 0u), kb = make_uint4(0u, 0u, 0u, 0u);
                        if (BK == 4) {
                            ka = *reinterpret_cast<const uint4 *>(kt + lane * 16);
                            kb = *reinterpret_cast<const uint4 *>(kt + 512 + lane * 16);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint2 kw0;
                            if (BK == 4)
                                kw0 = i == 0 ? make_uint2(ka.x, ka.y) : i == 1 ? make_uint2(ka.z, ka.w)
                                    : i == 2 ? make_uint2(kb.x, kb.y) : make_uint2(kb.z, kb.w);
                            else
                                kw0 = *reinterpret_cast<const uint2 *>(kt + 512 * (i >> 1) + lane * 16 + 8 * (i & 1));
                            // BK = 4: the plane-1 words of k-steps 2i, 2i+1, loaded where used (registers)
                            uint2 kw1 = make_uint2(0u, 0u);
                            if (BK == 4)
                                kw1 = *reinterpret_cast<const uint2 *>(kt + 1024 + 512 * (i >> 1) + lane * 16 + 8 * (i & 1));
                            const uint4 a = *reinterpret_cast<const uint4 *>(&S.qhi[hB][16 * i + 4 * r]);
                            const uint4 l = *reinterpret_cast<const uint4 *>(&S.qlo[hB][16 * i + 4 * r]);
                            const uint4 sv = *reinterpret_cast<const uint4 *>(ksz + (4 * i + r) * 8);
                            const uint4 zv = *reinterpret_cast<const uint4 *>(ksz + KVQ_D + (4 * i + r) * 8);
                            const uint4 qo = *reinterpret_cast<const uint4 *>(qown + 16 * i + 4 * r);
                            if (!ZMMA) {
                                // CUDA-core form: lane (q, r) adds its head hB's products over the lane's
                                // channels of k-steps 2i, 2i+1 (hi lanes the first, lo lanes the second)
                                const int k = 2 * i + (xB ? 1 : 0);
                                const uint2 zz = make_uint2(xB ? zv.z : zv.x, xB ? zv.w : zv.y);
                                const float4 qa = *reinterpret_cast<const float4 *>(&S.qz[hB][k * 16 + 4 * r]);
                                z0[0] = fmaf(qa.x, h2f(lo16(zz.x)), z0[0]);
                                z0[0] = fmaf(qa.y, h2f(hi16(zz.x)), z0[0]);
                                z0[0] = fmaf(qa.z, h2f(lo16(zz.y)), z0[0]);
                                z0[0] = fmaf(qa.w, h2f(hi16(zz.y)), z0[0]);
                            } else if (i & 1) {
                                mma16816(z1, zv.x, zv.x, zv.y, zv.y, qo.x, qo.y);
                                mma16816(z1, zv.z, zv.z, zv.w, zv.w, qo.z, qo.w);
                            } else {
                                mma16816(z0, zv.x, zv.x, zv.y, zv.y, qo.x, qo.y);
                                mma16816(z0, zv.z, zv.z, zv.w, zv.w, qo.z, qo.w);
                            }
                            const uint32_t bk[4] = {split_prod(a.x, l.x, sv.x, xB), split_prod(a.y, l.y, sv.y, xB),
                                                    split_prod(a.z, l.z, sv.z, xB), split_prod(a.w, l.w, sv.w, xB)};
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t w = kk ? kw0.y : kw0.x, w4 = w >> 4;
                                uint32_t a0l, a0h, a1l, a1h, a2l, a2h, a3l, a3h;
                                if (BK == 2) {
                                    e4m3x4_f16x2(w & 0x03030303u, a0l, a0h);
                                    e4m3x4_f16x2(w & 0x0C0C0C0Cu, a1l, a1h);
                                    e4m3x4_f16x2(w4 & 0x03030303u, a2l, a2h);
                                    e4m3x4_f16x2(w4 & 0x0C0C0C0Cu, a3l, a3h);
                                } else {
                                    // a nibble in bits 0-3 is the e4m3 pattern of code * 2^-9 (exact, linear)
                                    e4m3x4_f16x2(w & 0x0F0F0F0Fu, a0l, a0h);
                                    e4m3x4_f16x2(w4 & 0x0F0F0F0Fu, a1l, a1h);
                                    const uint32_t w1 = kk ? kw1.y : kw1.x;
                                    e4m3x4_f16x2(w1 & 0x0F0F0F0Fu, a2l, a2h);
                                    e4m3x4_f16x2((w1 >> 4) & 0x0F0F0F0Fu, a3l, a3h);
                                }
                                mma16816(s0, a0l, a1l, a0h, a1h, bk[2 * kk], bk[2 * kk + 1]);
                                mma16816(s1, a2l, a3l, a2h, a3h, bk[2 * kk], bk[2 * kk + 1]);
                            }
                        }
                    }
                    // ---- logits of head r, tokens q, q+8, q+16, q+24; online softmax ----
                    const float f9 = unsig * 512.f, f7 = BK == 4 ? f9 : unsig * 128.f;
                    float zr;
                    if (ZMMA) {
                        zr = ((z0[0] + z1[0]) + (z0[1] + z1[1])) * unsig;
                    } else {
                        // the 8 lanes of head hB hold its partial dots; head r's sum sits in lane 8r
                        float zp = z0[0];
                        zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 1);
                        zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 2);
                        zp += __shfl_xor_sync(0xFFFFFFFFu, zp, 4);
                        zr = __shfl_sync(0xFFFFFFFFu, zp, 8 * r);
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
                        for (int i = 0; i < NGV; ++i) vzc[i] *= sc;
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
                    // token 16k + 8hk + 4e + j (k-step k, m-row pair index 2j + e + 8hk) at
                    // position 16k + 8hk + 2j + e: each B register's two tokens are adjacent
                    float *pb = S.pbuf[warp];
#pragma unroll
                    for (int i = 0; i < 4; ++i) pb[r * PB_ROW + 8 * i + 2 * (q & 3) + (q >> 2)] = pr[i];
                    const uint32_t *vsz = reinterpret_cast<const uint32_t *>(st + GG::KC + GG::KSZ + GG::VC) +
                                          warp * 32 * NGV;
                    if (!ZMMA) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t row[NGV];
                            load_row<NGV>(vsz + (q + 8 * i) * NGV, row);
#pragma unroll
                            for (int j = 0; j < NGV; ++j) vzc[j] = fmaf(pr[i], h2f(hi16(row[j])), vzc[j]);
                        }
                    }
                    __syncwarp();
                    // ---- values: two 16-token k-steps x eight 16-channel m-tiles; k-column 2j + e + 8hk of
                    //      k-step k is token 16k + 8hk + 4e + j (rows of one load on distinct banks) ----
                    const uint8_t *vc = st + GG::KC + GG::KSZ + warp * 32 * (KVQ_D * BV / 8);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const int t0 = 16 * ks + r;             // tokens t0, t0+4 | t0+8, t0+12
                        // B: p_(hB, t) s_(t, j)
                        const float2 pa = *reinterpret_cast<const float2 *>(&pb[hB * PB_ROW + 16 * ks + 2 * r]);
                        const float2 pc = *reinterpret_cast<const float2 *>(&pb[hB * PB_ROW + 16 * ks + 8 + 2 * r]);
                        const uint32_t pha = split_pair(pa.x, pa.y, false), pla = split_pair(pa.x, pa.y, true);
                        const uint32_t phc = split_pair(pc.x, pc.y, false), plc = split_pair(pc.x, pc.y, true);
                        if (ZMMA) {
                            // value zero-point product: A rows hold z of group jz for the k-step's tokens (the
                            // high halves of the (s, z) words), B the lane's part of p
                            const uint32_t za = prmt(vsz[t0 * NGV + jz], vsz[(t0 + 4) * NGV + jz], 0x7632u);
                            const uint32_t zc = prmt(vsz[(t0 + 8) * NGV + jz], vsz[(t0 + 12) * NGV + jz], 0x7632u);
                            mma16816(vzacc, za, za, zc, zc, xB ? pla : pha, xB ? plc : phc);
                        }
                        uint32_t bv0[NGV], bv1[NGV];
                        {
                            uint32_t ra[NGV], rb[NGV], rc[NGV], rd[NGV];
                            load_row<NGV>(vsz + t0 * NGV, ra);
                            load_row<NGV>(vsz + (t0 + 4) * NGV, rb);
                            load_row<NGV>(vsz + (t0 + 8) * NGV, rc);
                            load_row<NGV>(vsz + (t0 + 12) * NGV, rd);
#pragma unroll
                            for (int j = 0; j < NGV; ++j) {
                                bv0[j] = split_prod(pha, pla, prmt(ra[j], rb[j], 0x5410u), xB);
                                bv1[j] = split_prod(phc, plc, prmt(rc[j], rd[j], 0x5410u), xB);
                            }
                        }
                        if (BV == 4) {
                            // the 4-bit value tile: lane 4q + r's 32 bytes of k-step ks are words 2m + w, m-tile m
                            // (channels 16m + q | + 8) in the low nibbles and m-tile m + 4 in the high nibbles, tokens
                            // t0, t0+4 (w = 0: k-columns 2r, 2r+1) and t0+8, t0+12 (w = 1: 2r+8, 2r+9)
                            const uint4 va = *reinterpret_cast<const uint4 *>(vc + ks * 1024 + lane * 32);
                            const uint4 vb4 = *reinterpret_cast<const uint4 *>(vc + ks * 1024 + lane * 32 + 16);
                            const uint32_t vw[8] = {va.x, va.y, va.z, va.w, vb4.x, vb4.y, vb4.z, vb4.w};
#pragma unroll
                            for (int m = 0; m < 4; ++m) {
                                const uint32_t x0 = vw[2 * m], x1 = vw[2 * m + 1];
                                const int jl = (16 * m) / (KVQ_D / NGV), jh = (16 * (m + 4)) / (KVQ_D / NGV);
                                uint32_t a0, a1, a2, a3;
                                e4m3x4_f16x2(x0 & 0x0F0F0F0Fu, a0, a1);
                                e4m3x4_f16x2(x1 & 0x0F0F0F0Fu, a2, a3);
                                mma16816(vacc[m], a0, a1, a2, a3, bv0[jl], bv1[jl]);
                                e4m3x4_f16x2((x0 >> 4) & 0x0F0F0F0Fu, a0, a1);
                                e4m3x4_f16x2((x1 >> 4) & 0x0F0F0F0Fu, a2, a3);
                                mma16816(vacc[m + 4], a0, a1, a2, a3, bv0[jh], bv1[jh]);
                            }
                        } else {
                            // m-tile 2g + pp, rows q | q + 8: channels 32g + 4q + 2pp + 0 | 1 (bit positions 2pp and
                            // 2pp + 1 of byte 8g + q); the value tile stores, for lane 4q + r, that byte of the
                            // tokens t0, t0+4 | t0+8, t0+12 as word g of its 16-byte chunk: the A registers of both
                            // m-tiles of group g
                            const uint4 v4 = *reinterpret_cast<const uint4 *>(vc + ks * 512 + lane * 16);
                            const uint32_t vx[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                            for (int g8 = 0; g8 < 4; ++g8) {
                                const uint32_t X = vx[g8];
                                const uint32_t X4 = X >> 4;
                                const int j = (32 * g8) / (KVQ_D / NGV);          // value group of both m-tiles
                                uint32_t a0, a1, a2, a3;
                                e4m3x4_f16x2(X & 0x03030303u, a0, a2);
                                e4m3x4_f16x2(X & 0x0C0C0C0Cu, a1, a3);
                                mma16816(vacc[2 * g8], a0, a1, a2, a3, bv0[j], bv1[j]);
                                e4m3x4_f16x2(X4 & 0x03030303u, a0, a2);
                                e4m3x4_f16x2(X4 & 0x0C0C0C0Cu, a1, a3);
                                mma16816(vacc[2 * g8 + 1], a0, a1, a2, a3, bv0[j], bv1[j]);
                            }
                        }
                    }
                    __syncwarp();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
            // ---- warp state (head r) -> shared memory ----
            float l_w = l_part;
            l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 4);
            l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 8);
            l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 16);
            float vz[NGV];
            if (ZMMA) {
                // group j's zero-point sum of head r sits in the lanes with q % NGV == j
                const float vzs = vzacc[0] + vzacc[1];
#pragma unroll
                for (int j = 0; j < NGV; ++j) vz[j] = __shfl_sync(0xFFFFFFFFu, vzs, 4 * j + r);
            } else {
#pragma unroll
                for (int j = 0; j < NGV; ++j) {
                    vz[j] = vzc[j];
                    vz[j] += __shfl_xor_sync(0xFFFFFFFFu, vz[j], 4);
                    vz[j] += __shfl_xor_sync(0xFFFFFFFFu, vz[j], 8);
                    vz[j] += __shfl_xor_sync(0xFFFFFFFFu, vz[j], 16);
                }
            }
            float *acc = S.st_acc[warp][r];
            if (BV == 4) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int j = (16 * mt) / (KVQ_D / NGV);
                    acc[16 * mt + q] = fmaf(vacc[mt][0] + vacc[mt][1], 512.f, vz[j]);
                    acc[16 * mt + q + 8] = fmaf(vacc[mt][2] + vacc[mt][3], 512.f, vz[j]);
                }
            } else {
                // rows q of both m-tiles of group g carry codes x 2^-9, rows q + 8 codes x 2^-7
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    const int j = (32 * g8) / (KVQ_D / NGV);
                    *reinterpret_cast<float4 *>(&acc[32 * g8 + 4 * q]) =
                        make_float4(fmaf(vacc[2 * g8][0] + vacc[2 * g8][1], 512.f, vz[j]),
                                    fmaf(vacc[2 * g8][2] + vacc[2 * g8][3], 128.f, vz[j]),
                                    fmaf(vacc[2 * g8 + 1][0] + vacc[2 * g8 + 1][1], 512.f, vz[j]),
                                    fmaf(vacc[2 * g8 + 1][2] + vacc[2 * g8 + 1][3], 128.f, vz[j]));
                }
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


// 2 <= g <= 4 heads per kv head in one unit, or an even g <= 8 in two units of g / 2 heads (the second
// unit of a kv head reads the same stages, mostly from L2: its units are neighbours in the unit order);
// any value group at 2/2 bits; with a 4-bit width the value group must be 32 channels (other
// 4-bit configurations run on the per-head kernel)
int kivi_gqa_units_per_kv_head(const kvq_config *cfg) {
    const int g = cfg->n_q_heads / cfg->n_kv_heads;
    return g > GMAX ? 2 : 1;
}

bool kivi_value_tiles(const kvq_config *cfg) { return kivi_gqa_supported(cfg); }

bool kivi_gqa_supported(const kvq_config *cfg) {
    const int g = cfg->n_q_heads / cfg->n_kv_heads;
    if (g < 2 || g > 2 * GMAX || (g > GMAX && g % 2 != 0)) return false;
    if (cfg->bits_k == 2 && cfg->bits_v == 2) return true;
    return cfg->group_v == 32;
}

template <int NGV, int BK, int BV, int NST>
static cudaError_t launch_gqa_variant(const Params &P, int64_t grid, cudaStream_t st) {
    const size_t smem = sizeof(SmemG<BK, BV, NST>);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(kivi_decode_gqa_kernel<NGV, BK, BV, NST>, smem, attr_done)) return e;
    kivi_decode_gqa_kernel<NGV, BK, BV, NST><<<(unsigned)grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_decode_kivi_gqa(const kvq_config *cfg, const KiviSrc &c, const void *q, const DecodePlan &p,
                                   void *ws, cudaStream_t st) {
    Params P = kivi_params(cfg, c, q, p, ws);
    if (!P.err) return cudaErrorInvalidDevicePointer;
    P.vsub = kivi_gqa_units_per_kv_head(cfg);
    P.gu = P.gall / P.vsub;
    const int64_t n_units = (int64_t)c.batch * cfg->n_kv_heads * P.vsub * p.splits;
    int64_t grid = (int64_t)num_sms() * 3;
    if (grid > n_units) grid = n_units;
    const int ngv = P.ngv;
    // 2/2 bits: three 12 KiB stages; with 4-bit codes (Gv = 32 only) two stages of up to 20 KiB
    if (cfg->bits_k == 2 && cfg->bits_v == 2) {
        if (ngv == 4) return launch_gqa_variant<4, 2, 2, 3>(P, grid, st);
        if (ngv == 2) return launch_gqa_variant<2, 2, 2, 3>(P, grid, st);
        return launch_gqa_variant<1, 2, 2, 3>(P, grid, st);
    }
    if (cfg->bits_k == 4 && cfg->bits_v == 4) return launch_gqa_variant<4, 4, 4, 2>(P, grid, st);
    if (cfg->bits_k == 4) return launch_gqa_variant<4, 4, 2, 2>(P, grid, st);
    return launch_gqa_variant<4, 2, 4, 2>(P, grid, st);
}

}  // namespace kvq
