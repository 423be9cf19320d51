// a3: KIVI split-KV decode attention, stage 1.
//
// Math (KIVI Eq. 3 with the dequantization folded out of the inner loops):
//   score_t = alpha * sum_c q_c (s_cg code_ct + z_cg)
//           = sum_c (alpha q_c s_cg) code_ct + alpha sum_c q_c z_cg
//   o_c     = sum_t p_t (s_tj code_tc + z_tj)
//           = sum_t (p_t s_tj) code_tc + sum_t p_t z_tj
// with alpha = sm_scale * log2(e) (softmax in base 2).
// Keys: the weights alpha q_c s_cg of a 32-token group are put in 22-bit
// fixed point against the group's largest |weight| (one power-of-two scale
// per tile) and split into three bytes; a packed word of key codes, masked
// in place, is four unsigned bytes code * 2^(b j) (b the code width, j the
// token's slot in the byte), so dp4a (four byte products summed into an
// int32) multiplies four channels' codes by one weight byte exactly.  Three
// dp4a per mask (one per weight byte) and the integer sums are exact; the
// only key rounding is the weights' fixed-point rounding (at most 2^-22 of
// the group's largest) and the final int -> fp32 conversion.  dp4a issues on
// the FMA-heavy pipe, beside the ALU pipe that the masks load (two LOP3 and
// one fma.rn.f32x2 per pair of codes loaded the ALU pipe alone: the dp4a form
// measured 9% faster on the MHA decode layer).
// Values: a 2-bit code masked in place out of its packed word, read as an
// fp32 bit pattern, is the denormal code * 2^(k-149) (k = its bit position,
// kept below the exponent field), so one LOP3 makes an exact fp32 operand
// and a packed fma.rn.f32x2 multiplies it by p_t s_tj pre-scaled per bit
// position (value_token_accum): the value products are exact in fp32 (s_tj
// code cancels against the zero point when the token's range is wide, so an
// fp16 weight would lose 2^-12 of a term much larger than the result).
// Powers of two are removed once per unit.
//
// Work decomposition: a persistent grid walks the (batch row, query head,
// split) units round-robin.  A producer warp streams every unit's 128-token
// stages (key codes, key (s, z), value codes, value (s, z): 12 KiB at
// G = Gv = 32) with 1-D bulk async copies (cp.async.bulk, the TMA engine)
// into a 3-slot shared-memory ring guarded by mbarriers, without pausing at
// unit boundaries; four consumer warps each take one 32-token tile of a
// stage.  The last split of every row is a residual unit: tokens whose key
// or value is not quantized (the fp16 residual, and any tile cut by a segment
// boundary), 32 per warp straight from global memory with every load of a
// block in flight together.  Each warp keeps an online softmax state per
// unit; the CTA merges the four warp states and writes (o_s, lse_s).
#include "kvq_kivi.cuh"

namespace kvq {

namespace {

constexpr int QK_ROW = 36;                // 32 channels + 4 floats of padding (bank spread)

template <int BK, int BV, int NSTAGE>
struct Smem {
    uint8_t stage[NSTAGE][Geo<BK, BV>::BYTES];
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    uint32_t qk[NCWARP][4 * QK_ROW];      // per-warp key weight bytes: row tq, (k: byte 0, 1, 2 of 4 channels, pad)
    float st_acc[NCWARP][KVQ_D];
    float st_m[NCWARP];
    float st_l[NCWARP];
    int abort_flag;                       // raised by a consumer warp whose wait gave up (last: the
                                          // members before it keep their 16-byte alignment)
};
// members read with 16-byte vector loads stay 16-byte aligned
using Smem_223 = Smem<2, 2, 3>;
using Smem_442 = Smem<4, 4, 2>;
static_assert(offsetof(Smem_223, qk) % 16 == 0 && offsetof(Smem_223, st_acc) % 16 == 0 &&
                  offsetof(Smem_442, qk) % 16 == 0 && offsetof(Smem_442, st_acc) % 16 == 0,
              "16-byte aligned shared-memory tables");

// Warp maximum of a float in one redux instruction: the bit patterns are
// mapped to unsigned integers in the floats' order (negative patterns
// complemented, non-negative ones given the top bit) and back.
__device__ __forceinline__ float warp_max_redux(float v) {
    uint32_t b = __float_as_uint(v);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    b = __reduce_max_sync(0xFFFFFFFFu, b);
    return __uint_as_float((b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b);
}

// Online-softmax update of a warp state with one logit per lane (-inf for
// empty lanes): returns p = 2^(logit - m) and rescales on a new maximum.
__device__ __forceinline__ float softmax_tile(float logit, float &m_run, float &l_part, float &vbias,
                                              unsigned long long vacc2[16]) {
    const float mt = warp_max_redux(logit);
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

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Fixed-point exponent fx of a group whose largest |weight| is wm: wm 2^fx
// lies in [2^21, 2^22), so every rounded weight is below 2^22 in magnitude
// and its top byte (bits 16-23, two's complement) is a signed byte in
// [-64, 64].  Clamped so that 2^fx and 2^-(fx + 6) stay normal fp32.
__device__ __forceinline__ int key_fixed_exp(float wm) {
    const int ex = (int)((__float_as_uint(wm) >> 23) & 255u);    // biased exponent, 0 for 0 and denormals
    return max(-100, min(100, 148 - ex));
}
// Four channels' weights in fixed point (rint(w 2^fx)), as three words of
// bytes: word i holds byte i of each channel's two's-complement value
// (channel order = the code word's byte order).
__device__ __forceinline__ uint4 key_weight_bytes(const float w[4], float scale) {
    const int w0 = __float2int_rn(w[0] * scale), w1 = __float2int_rn(w[1] * scale);
    const int w2 = __float2int_rn(w[2] * scale), w3 = __float2int_rn(w[3] * scale);
    uint32_t t01, t23, u01, u23, b0, b1, b2;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(t01) : "r"(w0), "r"(w1));   // w0.b0 w1.b0 w0.b1 w1.b1
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(t23) : "r"(w2), "r"(w3));
    asm("prmt.b32 %0, %1, %2, 0x0062;" : "=r"(u01) : "r"(w0), "r"(w1));   // w0.b2 w1.b2
    asm("prmt.b32 %0, %1, %2, 0x0062;" : "=r"(u23) : "r"(w2), "r"(w3));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(b0) : "r"(t01), "r"(t23));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(b1) : "r"(t01), "r"(t23));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(b2) : "r"(u01), "r"(u23));
    return make_uint4(b0, b1, b2, 0u);
}

}  // namespace

// BK-bit keys and BV-bit values (2 or 4) in an NSTAGE-slot ring.
template <int BK, int BV, int NSTAGE>
__global__ void __launch_bounds__(32 * (NCWARP + 1), 4) kivi_decode_kernel(Params P) {
    using GG = Geo<BK, BV>;
    constexpr int CPB = 8 / BK;                    // key codes per byte
    constexpr int NPL = BK / 2;                    // 1024-byte planes per 32-token key tile
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<BK, BV, NSTAGE> &S = *reinterpret_cast<Smem<BK, BV, NSTAGE> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_units = P.B * P.Hq * P.splits;
    const int G = P.G, Gv = P.Gv;

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
        // ---------------- producer: one stream of stages across all units ----------------
        if (lane == 0) kivi_produce<NSTAGE, false, BK, BV>(P, P.Hq, S.stage, S.full, S.empty, &S.abort_flag);
        return;
    }

    // ---------------- consumers ----------------
    const int tq = lane & 3;                       // key mapping: lane = 4*(token quad) + channel block
    const int ts = lane >> 2, jg = lane & 3;       // value mapping: token slot, channel block of 32
    const int gl = (32 * warp) / G;                // key group of this warp's tile within a stage
    const int ngv = P.ngv;
    const int jv = (32 * jg) / Gv;                 // value (s, z) group of this lane's channels
    bool ok = true;
    int sg = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = unit_of(P, u, P.Hq);
        float qa[4];
        const uint16_t *qrow = P.q + ((int64_t)U.b * P.Hq + U.hq) * KVQ_D;
        {
            const uint2 qv = *reinterpret_cast<const uint2 *>(qrow + 4 * lane);
            qa[0] = h2f(lo16(qv.x)) * P.alpha;
            qa[1] = h2f(hi16(qv.x)) * P.alpha;
            qa[2] = h2f(lo16(qv.y)) * P.alpha;
            qa[3] = h2f(hi16(qv.y)) * P.alpha;
        }
        if (U.residual) {
            // ---- residual unit ----
            float m_run, l_part, racc[4];
            kivi_residual(P, U, qa, warp, lane, racc, m_run, l_part);
            const float l_w = warp_sum(l_part);
            *reinterpret_cast<float4 *>(&S.st_acc[warp][4 * lane]) = make_float4(racc[0], racc[1], racc[2], racc[3]);
            if (lane == 0) {
                S.st_m[warp] = m_run;
                S.st_l[warp] = l_w;
            }
        } else {
            // lane writes weight-table entries 4*lane..4*lane+3: chunk row r = lane/8, word k = lane%8,
            // channels 16k + 2r + {0, 1, 8, 9}; query pre-scaled by the byte-parity power of two
            float qf[4];
            {
                const int c0 = 16 * (lane & 7) + 2 * (lane >> 3);
                const uint32_t q01 = *reinterpret_cast<const uint32_t *>(qrow + c0);
                const uint32_t q89 = *reinterpret_cast<const uint32_t *>(qrow + c0 + 8);
                qf[0] = h2f(lo16(q01)) * P.alpha;
                qf[1] = h2f(hi16(q01)) * P.alpha;
                qf[2] = h2f(lo16(q89)) * P.alpha;
                qf[3] = h2f(hi16(q89)) * P.alpha;
            }
            float m_run = -INFINITY, l_part = 0.f, vbias = 0.f;
            unsigned long long vacc2[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) vacc2[i] = 0ull;
            for (int s = 0; s < U.nstages; ++s, ++sg) {
                const int slot = sg % NSTAGE;
                ok = consumer_stage_wait(&S.full[slot], (sg / NSTAGE) & 1, P.err, KIVI_WAIT_LIMIT(P), ok, &S.abort_flag);
                const int tile = s * NCWARP + warp;
                if (ok && tile < U.nT) {
                    const uint8_t *st = S.stage[slot];
                    const uint16_t *ksz = reinterpret_cast<const uint16_t *>(st + GG::KC) + gl * 2 * KVQ_D;
                    // ---- this group's key weights alpha q s in 22-bit fixed point, and alpha sum q z ----
                    const int si = (((lane & 7) >> 1) * 4 + (lane >> 3)) * 8 + (lane & 1) * 4;
                    const uint2 sv = *reinterpret_cast<const uint2 *>(ksz + si);
                    const uint2 zv = *reinterpret_cast<const uint2 *>(ksz + KVQ_D + si);
                    const float w[4] = {qf[0] * h2f(lo16(sv.x)), qf[1] * h2f(hi16(sv.x)), qf[2] * h2f(lo16(sv.y)),
                                        qf[3] * h2f(hi16(sv.y))};
                    // the zero-point dot, and the largest |weight| (non-negative floats order as their bits)
                    const float cb = warp_sum(qf[0] * h2f(lo16(zv.x)) + qf[1] * h2f(hi16(zv.x)) +
                                              qf[2] * h2f(lo16(zv.y)) + qf[3] * h2f(hi16(zv.y)));
                    const float wm = __uint_as_float(__reduce_max_sync(
                        0xFFFFFFFFu, __float_as_uint(fmaxf(fmaxf(fabsf(w[0]), fabsf(w[1])), fmaxf(fabsf(w[2]), fabsf(w[3]))))));
                    const int fx = key_fixed_exp(wm);
                    *reinterpret_cast<uint4 *>(&S.qk[warp][(lane >> 3) * QK_ROW + 4 * (lane & 7)]) =
                        key_weight_bytes(w, __int_as_float((127 + fx) << 23));
                    __syncwarp();
                    // ---- key codes: tokens q + 8j (q = lane/4) x channels 16k + 2tq + {0,1,8,9};
                    //      token j sits in plane j / CPB at bits BK * (j % CPB) ----
                    const uint8_t *kt = st + warp * 512 * BK;
                    uint32_t kw[NPL][8];
#pragma unroll
                    for (int pl = 0; pl < NPL; ++pl) {
                        const uint4 ka = *reinterpret_cast<const uint4 *>(kt + pl * 1024 + lane * 16);
                        const uint4 kb = *reinterpret_cast<const uint4 *>(kt + pl * 1024 + 512 + lane * 16);
                        kw[pl][0] = ka.x; kw[pl][1] = ka.y; kw[pl][2] = ka.z; kw[pl][3] = ka.w;
                        kw[pl][4] = kb.x; kw[pl][5] = kb.y; kw[pl][6] = kb.z; kw[pl][7] = kb.w;
                    }
                    const uint4 *qd = reinterpret_cast<const uint4 *>(&S.qk[warp][tq * QK_ROW]);
                    int acc[4][3];                                              // token j, weight byte
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 d = qd[k];                                  // channels 16k + 2tq + {0,1,8,9}
#pragma unroll
                        for (int pl = 0; pl < NPL; ++pl) {
#pragma unroll
                            for (int jj = 0; jj < CPB; ++jj) {
                                const int j = pl * CPB + jj;
                                const uint32_t x = kw[pl][k] & ((((1u << BK) - 1) * 0x01010101u) << (BK * jj));
                                acc[j][0] = dp4a_uu(x, d.x, acc[j][0]);
                                acc[j][1] = dp4a_uu(x, d.y, acc[j][1]);
                                acc[j][2] = dp4a_us(x, d.z, acc[j][2]);
                            }
                        }
                    }
                    // weight bytes 0 + 1 fit an int32 (< 2^29); the sum is code * 2^(BK (j % CPB)) * W 2^fx
                    float a[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) a[j] = fmaf((float)acc[j][2], 65536.f, (float)(acc[j][0] + (acc[j][1] << 8)));
                    // transpose-reduce over the 4 lanes of the quad: lane keeps token q + 8tq
                    float score;
                    {
                        const bool h2 = (tq & 2) != 0;
                        float k0 = h2 ? a[2] : a[0], k1 = h2 ? a[3] : a[1];
                        k0 += __shfl_xor_sync(0xFFFFFFFFu, h2 ? a[0] : a[2], 2);
                        k1 += __shfl_xor_sync(0xFFFFFFFFu, h2 ? a[1] : a[3], 2);
                        const bool h1 = (tq & 1) != 0;
                        score = (h1 ? k1 : k0) + __shfl_xor_sync(0xFFFFFFFFu, h1 ? k0 : k1, 1);
                    }
                    const float logit = fmaf(score, __int_as_float((127 - fx - BK * (tq % CPB)) << 23), cb);
                    const float p = softmax_tile(logit, m_run, l_part, vbias, vacc2);
                    // ---- values: 4 passes of 8 tokens; lane = (token slot ts, channel block jg) ----
                    const uint8_t *vc = st + GG::KC + GG::KSZ + warp * 32 * (KVQ_D * BV / 8);
                    const uint32_t *vsz = reinterpret_cast<const uint32_t *>(st + GG::KC + GG::KSZ + GG::VC) +
                                          warp * 32 * ngv;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int tau = 8 * r + ts;
                        const float pt = __shfl_sync(0xFFFFFFFFu, p, 4 * ts + r);   // token tau = ts + 8r
                        const uint32_t szt = vsz[tau * ngv + jv];
                        vbias += pt * h2f(hi16(szt));
                        if (BV == 2)
                            value_token_accum(*reinterpret_cast<const uint2 *>(vc + tau * (KVQ_D / 4) + jg * 8),
                                              pt * h2f(lo16(szt)), vacc2);
                        else
                            value_token_accum4(*reinterpret_cast<const uint4 *>(vc + tau * (KVQ_D / 2) + jg * 16),
                                               pt * h2f(lo16(szt)), vacc2);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }

            // ---- warp state -> shared memory (channel order) ----
            {
                const float l_w = warp_sum(l_part);
                float vb = vbias;
                vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 4);
                vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 8);
                vb += __shfl_xor_sync(0xFFFFFFFFu, vb, 16);
                // lane (ts, jg) writes channels 32jg + 4ts + i (i = 0..3) plus the zero-point term
                float4 w4 = value_block_reduce<BV>(vacc2, ts);
                w4.x += vb; w4.y += vb; w4.z += vb; w4.w += vb;
                *reinterpret_cast<float4 *>(&S.st_acc[warp][32 * jg + 4 * ts]) = w4;
                if (lane == 0) {
                    S.st_m[warp] = m_run;
                    S.st_l[warp] = l_w;
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
        // ---- merge the four warp states, write (o_s, lse_s) of the unit ----
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

template <int BK, int BV, int NST>
static cudaError_t launch_kivi_variant(const Params &P, int64_t grid, cudaStream_t st) {
    const size_t smem = sizeof(Smem<BK, BV, NST>);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(kivi_decode_kernel<BK, BV, NST>, smem, attr_done)) return e;
    kivi_decode_kernel<BK, BV, NST><<<(unsigned)grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_decode_kivi(const kvq_config *cfg, const KiviSrc &c, const void *q, const DecodePlan &p,
                               void *ws, cudaStream_t st) {
    Params P = kivi_params(cfg, c, q, p, ws);
    if (!P.err) return cudaErrorInvalidDevicePointer;
    const int64_t n_units = (int64_t)c.batch * cfg->n_q_heads * p.splits;
    int64_t grid = (int64_t)num_sms() * 4;
    if (grid > n_units) grid = n_units;
    // the ring holds 3 stages of 12 KiB at 2/2 bits (measured 1.5% faster than 4 on the MHA workload),
    // 3 of 16 KiB at 4/2 or 2/4, 2 of 20 KiB at 4/4 (4 CTAs per SM)
    if (cfg->bits_k == 2 && cfg->bits_v == 2) return launch_kivi_variant<2, 2, 3>(P, grid, st);
    if (cfg->bits_k == 4 && cfg->bits_v == 2) return launch_kivi_variant<4, 2, 3>(P, grid, st);
    if (cfg->bits_k == 2 && cfg->bits_v == 4) return launch_kivi_variant<2, 4, 3>(P, grid, st);
    return launch_kivi_variant<4, 4, 2>(P, grid, st);
}

}  // namespace kvq
