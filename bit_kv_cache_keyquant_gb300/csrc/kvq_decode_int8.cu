// a9: WitCert INT8 subtractive-dither decode attention, stage 1.
//
// K^ = s (code - xi) with s the block's per-channel fp16 scale and xi the
// Philox4x32-10 dither regenerated from (request, layer, kv head, token,
// channel) exactly as the write kernel drew it (WitCert sec. 6.1: the read
// side uses the same five-tuple Philox as the write side).  The active
// (incomplete) 256-token block stays fp16.
//
// The path is bound by integer ALU work (the Philox rounds), not HBM, so the
// kernel computes every dither once per element and shares it across all
// g <= 8 query heads of the kv head:
//   * one CTA per (batch row, kv head, split) unit of a persistent grid; a
//     producer warp streams 128-token stages (int8 K and V codes, 16 KiB
//     each, plus the block's K and V scales) with cp.async.bulk into a
//     2-slot mbarrier ring;
//   * a consumer warp owns 32 tokens of a stage; lane l owns channels
//     4l..4l+3, so one Philox call (counter word 1 = l) yields its four
//     dithers per token (the "four-output reuse");
//   * keys: per token, 8 head partials over the lane's 4 channels; for 4
//     tokens at a time each lane writes its 32 partials as one row of a
//     per-warp shared-memory block and then sums one column over the 32
//     rows, so that lane L holds head L%8 of token L/8 of the four;
//     per-head online softmax in base 2;
//   * values: the 8 head weights of each token are broadcast through shared
//     memory and accumulated into 8 x 4 fp32 accumulators per lane.
// The last split of every row covers the fp16 tail with the same tile code.
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int NSTAGE = 2;
constexpr int NCWARP = 4;
constexpr int STAGE_TOK = 32 * NCWARP;                 // 128 tokens
constexpr int CODES_BYTES = STAGE_TOK * KVQ_D;         // 16 KiB per side
constexpr int STAGE_BYTES = 2 * CODES_BYTES + 2 * KVQ_D * 2;
constexpr int GMAX = 8;

struct Smem {
    uint8_t stage[NSTAGE][STAGE_BYTES];
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    float pw[NCWARP][32][GMAX];            // per-warp softmax weights of the tile's 32 tokens
    union {                                // a warp's region: key partials inside a tile, its state at the unit end
        float st_acc[NCWARP][GMAX][KVQ_D];
        float red[NCWARP][32][32];
    };
    float st_m[NCWARP][GMAX];
    float st_l[NCWARP][GMAX];
    int abort_flag;                       // raised by a consumer warp whose wait gave up (last: the
                                          // members before it keep their 16-byte alignment)
};
static_assert(offsetof(Smem, pw) % 16 == 0 && offsetof(Smem, st_acc) % 16 == 0, "16-byte aligned tables");

struct Params {
    const int32_t *seq_len;
    const int32_t *req_id;
    const int8_t *k_codes, *v_codes;
    const uint16_t *k_scale, *v_scale, *k_tail, *v_tail;
    const uint16_t *q;
    float *ws_o, *ws_lse;
    unsigned *err;
    int B, Hq, Hkv, g, T, splits, chunk, blk_cap;
    int64_t cap;
    uint32_t ctr2_layer, k0, k1;
    uint32_t rk0[10], rk1[10];   // Philox round keys (k0 + r*0x9E3779B9, k1 + r*0xBB67AE85)
    float alpha;
};

struct Unit {
    int b, kvh, split, t0, t1, nq, L;
    bool residual;
    int64_t bk;
};

__device__ __forceinline__ Unit unit_of(const Params &P, int u) {
    Unit U;
    // split-major numbering (u = split * rows + row): every CTA's round-robin
    // share mixes all splits, whose lengths differ with the rows' lengths
    const int rows = P.B * P.Hkv;
    U.split = u / rows;
    const int row = u - U.split * rows;
    U.b = row / P.Hkv;
    U.kvh = row - U.b * P.Hkv;
    U.L = clamp_len(P.seq_len[U.b], (int)P.cap, P.err);
    const int ntail = ((U.L - 1) % P.T) + 1;
    U.nq = U.L - ntail;
    U.residual = U.split == P.splits - 1;
    if (U.residual) {
        U.t0 = U.nq;
        U.t1 = U.L;
    } else {
        U.t0 = U.split * P.chunk;
        U.t1 = max(U.t0, min(U.t0 + P.chunk, U.nq));
    }
    U.bk = (int64_t)U.b * P.Hkv + U.kvh;
    return U;
}

// Philox4x32-10 with the round keys taken from the kernel parameters (the
// same bijection as philox4x32_10: 32x32->64 products, xor with the round
// key; only the key schedule is precomputed).
__device__ __forceinline__ uint4 philox_rk(uint4 c, const uint32_t *rk0, const uint32_t *rk1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        unsigned long long pa, pb;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(pa) : "r"(c.x), "r"(0xD2511F53u));
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(pb) : "r"(c.z), "r"(0xCD9E8D57u));
        c = make_uint4((uint32_t)(pb >> 32) ^ c.y ^ rk0[r], (uint32_t)pb, (uint32_t)(pa >> 32) ^ c.w ^ rk1[r],
                       (uint32_t)pa);
    }
    return c;
}

// code - xi of the four channels 4*lane..4*lane+3 (codes: the int8 bytes of
// w), with the dither of counter word 0 = t (the token, or the slot) and
// word 3 = w3: xi = (r >> 8) 2^-24 - 1/2 exactly, so code - xi is
// (code + 1/2) - (r >> 8) 2^-24 before its one rounding, formed by one FMA
// (the same fp32 number as fl(code - xi)).
template <typename PP>
__device__ __forceinline__ void code_minus_dither4(const PP &P, uint32_t w, uint32_t c2, uint32_t w3, int t, int lane,
                                                   float d[4]) {
    const uint4 r = philox_rk(make_uint4((uint32_t)t, (uint32_t)lane, c2, w3), P.rk0, P.rk1);
    const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] = fmaf(__uint2float_rn(rr[i] >> 8), -0x1.0p-24f, (float)(int8_t)((w >> (8 * i)) & 0xFFu) + 0.5f);
}

// Per-lane attention state: output accumulators of the lane's four channels
// for all GMAX heads, as (head 2j, head 2j+1) pairs per channel, and the
// online-softmax state of head lane & 7.
struct HeadState {
    unsigned long long acc2[GMAX / 2][4];
    float m, l;
};

// alpha q of the g <= GMAX query heads of kv head kvh (q_row = the batch
// row's [Hq][D] queries) for this lane's four channels, as head pairs;
// heads >= g get weight 0
__device__ __forceinline__ void load_key_weights(const uint16_t *q_row, int kvh, int g, float alpha, int lane,
                                                 unsigned long long wk2[GMAX / 2][4]) {
    float qa[GMAX][4];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        const int hq = kvh * g + min(h, g - 1);
        const uint2 qv = *reinterpret_cast<const uint2 *>(q_row + (int64_t)hq * KVQ_D + 4 * lane);
        const float z = h < g ? alpha : 0.f;
        qa[h][0] = h2f(lo16(qv.x)) * z;
        qa[h][1] = h2f(hi16(qv.x)) * z;
        qa[h][2] = h2f(lo16(qv.y)) * z;
        qa[h][3] = h2f(hi16(qv.y)) * z;
    }
#pragma unroll
    for (int j = 0; j < GMAX / 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) wk2[j][i] = pack2f(qa[2 * j][i], qa[2 * j + 1][i]);
}

__device__ __forceinline__ void head_state_init(HeadState &H) {
    H.m = -INFINITY;
    H.l = 0.f;
#pragma unroll
    for (int j = 0; j < GMAX / 2; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) H.acc2[j][i] = 0ull;
}

// Merge the NCWARP consumer warps' states of one unit and write (o_s, lse_s)
// of its g query heads (workspace rows head_row0 .. head_row0 + g - 1).
template <typename SM>
__device__ __forceinline__ void write_unit(SM &S, const HeadState &H, float *ws_o, float *ws_lse, int64_t head_row0,
                                           int g, int splits, int split, int warp, int lane) {
    // ---- warp states -> shared memory ----
    __syncwarp();                        // the last tile's reads of this warp's reduction rows are done
    {
        float l_w = H.l;
        l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 8);
        l_w += __shfl_xor_sync(0xFFFFFFFFu, l_w, 16);
#pragma unroll
        for (int j = 0; j < GMAX / 2; ++j) {
            *reinterpret_cast<float4 *>(&S.st_acc[warp][2 * j][4 * lane]) =
                make_float4(lo2f(H.acc2[j][0]), lo2f(H.acc2[j][1]), lo2f(H.acc2[j][2]), lo2f(H.acc2[j][3]));
            *reinterpret_cast<float4 *>(&S.st_acc[warp][2 * j + 1][4 * lane]) =
                make_float4(hi2f(H.acc2[j][0]), hi2f(H.acc2[j][1]), hi2f(H.acc2[j][2]), hi2f(H.acc2[j][3]));
        }
        if (lane < GMAX) {
            S.st_m[warp][lane] = H.m;
            S.st_l[warp][lane] = l_w;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
    // ---- merge the four warp states per head: warp w writes heads w, w + 4 ----
    for (int h = warp; h < g; h += NCWARP) {
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
        const int64_t row = (head_row0 + h) * splits + split;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        *reinterpret_cast<float4 *>(ws_o + row * KVQ_D + 4 * lane) =
            make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
        if (lane == 0) ws_lse[row] = l > 0.f ? M + log2f(l) : -INFINITY;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * NCWARP) : "memory");
}

// One tile of n <= 32 tokens.  kfn(tt, kv[4]) / vfn(tt, vv[4]) return this
// lane's four dequantized channels of token tt of the tile; wk2[j][i] holds
// the key weights (alpha q) of heads 2j, 2j+1 for channel i.  KU key batches
// of four tokens and VU value tokens are unrolled together, so that more
// Philox chains are in flight (KU = 2, VU = 8 measured 871.7 -> 823.8 us on
// the block-INT8 workload, 1178.6 -> 1137.9 us on the slot-pool one).
template <int KU, int VU, typename KF, typename VF>
__device__ __forceinline__ void tile(int n, const unsigned long long wk2[GMAX / 2][4], KF kfn, VF vfn, HeadState &H,
                                     float (*pw)[GMAX], float (*red)[32], int lane) {
    // ---- keys: 8 batches of 4 tokens; per lane 4 x 8 head partials over its 4 channels, then a
    //      sum over all 32 lanes leaves lane L with token 4c + L/8, head L%8 ----
    float sc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) sc[c] = -INFINITY;
#pragma unroll KU
    for (int c4 = 0; c4 < 8; ++c4) {
        float v[32];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            float kv[4];
            kfn(min(4 * c4 + m, n - 1), kv);
#pragma unroll
            for (int j = 0; j < GMAX / 2; ++j) {
                unsigned long long d = 0ull;
#pragma unroll
                for (int i = 0; i < 4; ++i) d = ffma2(wk2[j][i], pack2f(kv[i], kv[i]), d);
                v[8 * m + 2 * j] = lo2f(d);
                v[8 * m + 2 * j + 1] = hi2f(d);
            }
        }
        // sum over the 32 lanes through shared memory: lane l stores its 32 partials as row l (16-byte
        // chunk k at k ^ (l & 7): four wavefronts a store), then lane L sums column L (conflict-free)
        __syncwarp();                                              // the previous batch's columns are read
#pragma unroll
        for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4 *>(&red[lane][4 * (k ^ (lane & 7))]) =
                make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        __syncwarp();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};                      // four chains of eight dependent adds
        const int col = lane & 3, chunk = lane >> 2;
#pragma unroll
        for (int l = 0; l < 32; ++l) acc[l & 3] += red[l][4 * (chunk ^ (l & 7)) + col];
        const float s = 4 * c4 + (lane >> 3) < n ? (acc[0] + acc[1]) + (acc[2] + acc[3]) : -INFINITY;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            if (c == c4) sc[c] = s;
    }
    // ---- online softmax of head lane & 7 (its tokens live in lanes h, h+8, h+16, h+24) ----
    float mt = sc[0];
#pragma unroll
    for (int c = 1; c < 8; ++c) mt = fmaxf(mt, sc[c]);
    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 8));
    mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 16));
    const float mnew = fmaxf(H.m, mt);
    const float scl = exp2f(H.m - mnew);
    H.m = mnew;
    H.l *= scl;
#pragma unroll
    for (int j = 0; j < GMAX / 2; ++j) {
        const unsigned long long sp =
            pack2f(__shfl_sync(0xFFFFFFFFu, scl, 2 * j), __shfl_sync(0xFFFFFFFFu, scl, 2 * j + 1));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            unsigned long long d;
            asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(H.acc2[j][i]), "l"(sp));
            H.acc2[j][i] = d;
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const float p = exp2f(sc[c] - mnew);
        H.l += p;
        pw[4 * c + (lane >> 3)][lane & 7] = p;
    }
    __syncwarp();
    // ---- values: lane = channels, head weights broadcast from shared memory ----
#pragma unroll VU
    for (int tt = 0; tt < 32; ++tt) {
        if (tt >= n) break;
        float vv[4];
        vfn(tt, vv);
        const float4 p0 = *reinterpret_cast<const float4 *>(&pw[tt][0]);
        const float4 p1 = *reinterpret_cast<const float4 *>(&pw[tt][4]);
        const unsigned long long pp[GMAX / 2] = {pack2f(p0.x, p0.y), pack2f(p0.z, p0.w), pack2f(p1.x, p1.y),
                                                 pack2f(p1.z, p1.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const unsigned long long vi = pack2f(vv[i], vv[i]);
#pragma unroll
            for (int j = 0; j < GMAX / 2; ++j) H.acc2[j][i] = ffma2(pp[j], vi, H.acc2[j][i]);
        }
    }
    __syncwarp();
}

}  // namespace

__global__ void __launch_bounds__(32 * (NCWARP + 1), 2) int8_decode_kernel(Params P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_units = P.B * P.Hkv * P.splits;

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
        if (lane == 0) {
            bool ok = true;
            int sg = 0;
            int armed[NSTAGE];
#pragma unroll
            for (int j = 0; j < NSTAGE; ++j) armed[j] = 0;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit U = unit_of(P, u);
                const int nst = U.residual ? 0 : (U.t1 - U.t0 + STAGE_TOK - 1) / STAGE_TOK;
                for (int s = 0; s < nst; ++s, ++sg) {
                    const int slot = sg % NSTAGE;
                    if (sg >= NSTAGE) ok = mbar_wait(&S.empty[slot], ((sg / NSTAGE) - 1) & 1, P.err);
                    ok = ok && !ring_aborted(&S.abort_flag);
                    if (!ok) break;
                    const int tok = U.t0 + s * STAGE_TOK;
                    const int nt = min(STAGE_TOK, U.t1 - tok);
                    const int blk = tok / P.T;
                    uint8_t *st = S.stage[slot];
                    ++armed[slot];
                    mbar_expect_tx(&S.full[slot], (uint32_t)(2 * nt * KVQ_D + 4 * KVQ_D));
                    bulk_g2s(st, P.k_codes + (U.bk * P.cap + tok) * KVQ_D, nt * KVQ_D, &S.full[slot]);
                    bulk_g2s(st + CODES_BYTES, P.v_codes + (U.bk * P.cap + tok) * KVQ_D, nt * KVQ_D, &S.full[slot]);
                    bulk_g2s(st + 2 * CODES_BYTES, P.k_scale + (U.bk * P.blk_cap + blk) * KVQ_D, 2 * KVQ_D,
                             &S.full[slot]);
                    bulk_g2s(st + 2 * CODES_BYTES + 2 * KVQ_D, P.v_scale + (U.bk * P.blk_cap + blk) * KVQ_D, 2 * KVQ_D,
                             &S.full[slot]);
                }
            }
            producer_drain<NSTAGE>(S.full, armed, P.err);
        }
        return;
    }

    const int g = P.g;
    bool ok = true;
    int sg = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const Unit U = unit_of(P, u);
        unsigned long long wk2[GMAX / 2][4];
        load_key_weights(P.q + (int64_t)U.b * P.Hq * KVQ_D, U.kvh, g, P.alpha, lane, wk2);
        HeadState H;
        head_state_init(H);
        const uint32_t c2 = P.ctr2_layer | (uint32_t)U.kvh;
        const uint32_t req = (uint32_t)P.req_id[U.b];
        if (U.residual) {
            const uint16_t *kt = P.k_tail + U.bk * (int64_t)P.T * KVQ_D + 4 * lane;
            const uint16_t *vt = P.v_tail + U.bk * (int64_t)P.T * KVQ_D + 4 * lane;
            const int T = P.T;
            for (int r0 = U.t0 + 32 * warp; r0 < U.t1; r0 += 32 * NCWARP) {
                const int n = min(32, U.t1 - r0);
                auto kfn = [=](int tt, float kv[4]) {
                    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(kt + (int64_t)((r0 + tt) % T) * KVQ_D));
                    kv[0] = h2f(lo16(x.x)); kv[1] = h2f(hi16(x.x)); kv[2] = h2f(lo16(x.y)); kv[3] = h2f(hi16(x.y));
                };
                auto vfn = [=](int tt, float vv[4]) {
                    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(vt + (int64_t)((r0 + tt) % T) * KVQ_D));
                    vv[0] = h2f(lo16(x.x)); vv[1] = h2f(hi16(x.x)); vv[2] = h2f(lo16(x.y)); vv[3] = h2f(hi16(x.y));
                };
                tile<2, 8>(n, wk2, kfn, vfn, H, S.pw[warp], S.red[warp], lane);
            }
        } else {
            const int nst = (U.t1 - U.t0 + STAGE_TOK - 1) / STAGE_TOK;
            for (int s = 0; s < nst; ++s, ++sg) {
                const int slot = sg % NSTAGE;
                ok = consumer_stage_wait(&S.full[slot], (sg / NSTAGE) & 1, P.err, KVQ_SPIN_LIMIT, ok, &S.abort_flag);
                const int tok = U.t0 + s * STAGE_TOK;
                const int r0 = tok + 32 * warp;
                const int n = min(32, U.t1 - r0);
                if (ok && n > 0) {
                    const uint8_t *st = S.stage[slot];
                    const uint8_t *kc = st + 32 * warp * KVQ_D + 4 * lane;
                    const uint8_t *vc = st + CODES_BYTES + 32 * warp * KVQ_D + 4 * lane;
                    const uint2 ks = *reinterpret_cast<const uint2 *>(st + 2 * CODES_BYTES + 8 * lane);
                    const uint2 vs = *reinterpret_cast<const uint2 *>(st + 2 * CODES_BYTES + 2 * KVQ_D + 8 * lane);
                    const float ks0 = h2f(lo16(ks.x)), ks1 = h2f(hi16(ks.x)), ks2 = h2f(lo16(ks.y)), ks3 = h2f(hi16(ks.y));
                    const float vs0 = h2f(lo16(vs.x)), vs1 = h2f(hi16(vs.x)), vs2 = h2f(lo16(vs.y)), vs3 = h2f(hi16(vs.y));
                    auto kfn = [=](int tt, float kv[4]) {
                        float d[4];
                        code_minus_dither4(P, *reinterpret_cast<const uint32_t *>(kc + tt * KVQ_D), c2, req, r0 + tt,
                                           lane, d);
                        kv[0] = ks0 * d[0];
                        kv[1] = ks1 * d[1];
                        kv[2] = ks2 * d[2];
                        kv[3] = ks3 * d[3];
                    };
                    auto vfn = [=](int tt, float vv[4]) {
                        float d[4];
                        code_minus_dither4(P, *reinterpret_cast<const uint32_t *>(vc + tt * KVQ_D), c2 | 0x10000u, req,
                                           r0 + tt, lane, d);
                        vv[0] = vs0 * d[0];
                        vv[1] = vs1 * d[1];
                        vv[2] = vs2 * d[2];
                        vv[3] = vs3 * d[3];
                    };
                    tile<2, 8>(n, wk2, kfn, vfn, H, S.pw[warp], S.red[warp], lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[slot]);
            }
        }
        write_unit(S, H, P.ws_o, P.ws_lse, (int64_t)U.b * P.Hq + U.kvh * g, g, P.splits, U.split, warp, lane);
    }
}

cudaError_t launch_decode_int8(const kvq_config *cfg, const kvq_int8_cache *c, const void *q, const DecodePlan &p,
                               void *ws, cudaStream_t st) {
    Params P;
    P.seq_len = c->seq_len;
    P.req_id = c->req_id;
    P.k_codes = static_cast<const int8_t *>(c->k_codes);
    P.v_codes = static_cast<const int8_t *>(c->v_codes);
    P.k_scale = static_cast<const uint16_t *>(c->k_scale);
    P.v_scale = static_cast<const uint16_t *>(c->v_scale);
    P.k_tail = static_cast<const uint16_t *>(c->k_tail);
    P.v_tail = static_cast<const uint16_t *>(c->v_tail);
    P.q = static_cast<const uint16_t *>(q);
    P.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_o);
    P.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_lse);
    P.err = device_error_ptr();
    P.B = c->batch;
    P.Hq = cfg->n_q_heads;
    P.Hkv = cfg->n_kv_heads;
    P.g = cfg->n_q_heads / cfg->n_kv_heads;
    P.T = cfg->int8_block;
    P.splits = p.splits;
    P.chunk = p.chunk;
    P.cap = c->max_seq_len;
    P.blk_cap = (c->max_seq_len + P.T - 1) / P.T;
    if (P.blk_cap < 1) P.blk_cap = 1;
    P.ctr2_layer = (uint32_t)c->layer << 17;
    P.k0 = (uint32_t)(c->seed & 0xFFFFFFFFu);
    P.k1 = (uint32_t)(c->seed >> 32);
    for (int r = 0; r < 10; ++r) {
        P.rk0[r] = P.k0 + (uint32_t)r * 0x9E3779B9u;
        P.rk1[r] = P.k1 + (uint32_t)r * 0xBB67AE85u;
    }
    P.alpha = sm_scale_of(cfg) * 1.4426950408889634f;
    if (!P.err) return cudaErrorInvalidDevicePointer;
    if (P.g > GMAX) return cudaErrorInvalidValue;
    const size_t smem = sizeof(Smem);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(int8_decode_kernel, smem, attr_done)) return e;
    const int64_t n_units = (int64_t)c->batch * cfg->n_kv_heads * p.splits;
    int64_t grid = (int64_t)num_sms() * 2;
    if (grid > n_units) grid = n_units;
    int8_decode_kernel<<<(unsigned)grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Token-granular INT8 over a slot pool (WitCert, SGLang storage subsection):
// token t of request b lives in slot table[b][t]; its codes are one 128-byte
// row of the pool and its scales one fp16 per Gc channels.  Same tile code as
// above; the producer warp gathers a stage's rows by slot: each of its 32
// lanes reads the slots of four tokens, copies their scales (plain loads, 2-8
// bytes) and slot ids into shared memory, arrives on the stage barrier with
// the byte count of its code rows and then issues those 128-byte bulk copies.
// Every token is quantized, so there is no fp16 tail and no residual unit.
// ---------------------------------------------------------------------------
namespace {

struct SmemT {
    uint8_t kc[NSTAGE][CODES_BYTES];
    uint8_t vc[NSTAGE][CODES_BYTES];
    uint16_t ks[NSTAGE][STAGE_TOK][4];     // per-token scales, D/Gc <= 4 used
    uint16_t vs[NSTAGE][STAGE_TOK][4];
    int32_t slot[NSTAGE][STAGE_TOK];
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    float pw[NCWARP][32][GMAX];
    union {
        float st_acc[NCWARP][GMAX][KVQ_D];
        float red[NCWARP][32][32];
    };
    float st_m[NCWARP][GMAX];
    float st_l[NCWARP][GMAX];
    int abort_flag;                       // raised by a consumer warp whose wait gave up (last: the
                                          // members before it keep their 16-byte alignment)
};
static_assert(offsetof(SmemT, pw) % 16 == 0 && offsetof(SmemT, st_acc) % 16 == 0, "16-byte aligned tables");

struct ParamsT {
    const int32_t *seq_len, *table;
    const int8_t *k_codes, *v_codes;
    const uint16_t *k_scale, *v_scale;
    const uint16_t *q;
    float *ws_o, *ws_lse;
    unsigned *err;
    int B, Hq, Hkv, g, splits, chunk, cap, n_slots, nsc, gshift;
    uint32_t ctr2_layer;
    uint32_t rk0[10], rk1[10];
    float alpha;
};

struct UnitT {
    int b, kvh, split, t0, t1;
};

__device__ __forceinline__ UnitT unit_of_t(const ParamsT &P, int u) {
    UnitT U;
    const int rows = P.B * P.Hkv;
    U.split = u / rows;
    const int row = u - U.split * rows;
    U.b = row / P.Hkv;
    U.kvh = row - U.b * P.Hkv;
    const int L = clamp_len(P.seq_len[U.b], P.cap, P.err);   // a length above the table's row: the full row
    U.t0 = U.split * P.chunk;
    U.t1 = max(U.t0, min(U.t0 + P.chunk, L));
    return U;
}

// nsc fp16 scales of one record (nsc = 4, 2 or 1; 8-, 4- or 2-byte aligned)
__device__ __forceinline__ uint2 load_scales(const uint16_t *p, int nsc) {
    if (nsc == 4) return __ldg(reinterpret_cast<const uint2 *>(p));
    if (nsc == 2) return make_uint2(__ldg(reinterpret_cast<const unsigned *>(p)), 0u);
    return make_uint2((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)), 0u);
}

}  // namespace

__global__ void __launch_bounds__(32 * (NCWARP + 1), 2) int8_token_decode_kernel(ParamsT P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SmemT &S = *reinterpret_cast<SmemT *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_units = P.B * P.Hkv * P.splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&S.full[i], 64);      // per producer lane: its slots and scales, then its code copies
            mbar_init(&S.empty[i], NCWARP);
        }
        S.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCWARP) {
        bool ok = true;
        int sg = 0;
        int armed[NSTAGE];
#pragma unroll
        for (int j = 0; j < NSTAGE; ++j) armed[j] = 0;
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const UnitT U = unit_of_t(P, u);
            const int nst = (U.t1 - U.t0 + STAGE_TOK - 1) / STAGE_TOK;
            const int32_t *trow = P.table + (int64_t)U.b * P.cap;
            for (int s = 0; s < nst; ++s, ++sg) {
                const int buf = sg % NSTAGE;
                if (sg >= NSTAGE) ok = mbar_wait(&S.empty[buf], ((sg / NSTAGE) - 1) & 1, P.err);
                ok = __all_sync(0xFFFFFFFFu, ok && !ring_aborted(&S.abort_flag));
                if (!ok) break;
                ++armed[buf];
                const int tok = U.t0 + s * STAGE_TOK;
                const int nt = min(STAGE_TOK, U.t1 - tok);
                int64_t rec[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = lane + 32 * j;
                    rec[j] = -1;
                    if (i < nt) {
                        int32_t sl = __ldg(trow + tok + i);
                        if (sl < 0 || sl >= P.n_slots) {   // a table entry outside the pool: read slot 0, flag it
                            atomicOr(P.err, KVQ_DEVICE_ERR_POOL);
                            sl = 0;
                        }
                        rec[j] = (int64_t)sl * P.Hkv + U.kvh;
                        S.slot[buf][i] = sl;
                        const uint2 a = load_scales(P.k_scale + rec[j] * P.nsc, P.nsc);
                        const uint2 b = load_scales(P.v_scale + rec[j] * P.nsc, P.nsc);
                        *reinterpret_cast<uint2 *>(&S.ks[buf][i][0]) = a;
                        *reinterpret_cast<uint2 *>(&S.vs[buf][i][0]) = b;
                    }
                }
                mbar_arrive(&S.full[buf]);                 // the slots and scales this lane stored
                // the tokens' code rows, 16 bytes per copy from every lane (no per-lane serialization of
                // bulk copies); the stage barrier counts this lane's arrival once all of them landed
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (rec[j] >= 0) {
                        const int i = lane + 32 * j;
                        const int8_t *kg = P.k_codes + rec[j] * KVQ_D, *vg = P.v_codes + rec[j] * KVQ_D;
#pragma unroll
                        for (int c = 0; c < KVQ_D / 16; ++c) {
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                                         ::"r"(smem_addr(S.kc[buf] + i * KVQ_D + 16 * c)), "l"(kg + 16 * c) : "memory");
                            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                                         ::"r"(smem_addr(S.vc[buf] + i * KVQ_D + 16 * c)), "l"(vg + 16 * c) : "memory");
                        }
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&S.full[buf]))
                             : "memory");
            }
        }
        // no copy may be in flight when the CTA exits
        producer_drain<NSTAGE>(S.full, armed, P.err);
        return;
    }

    const int g = P.g;
    const int gi = lane >> P.gshift;       // the lane's channel group
    bool ok = true;
    int sg = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const UnitT U = unit_of_t(P, u);
        unsigned long long wk2[GMAX / 2][4];
        load_key_weights(P.q + (int64_t)U.b * P.Hq * KVQ_D, U.kvh, g, P.alpha, lane, wk2);
        HeadState H;
        head_state_init(H);
        const uint32_t c2 = P.ctr2_layer | (uint32_t)U.kvh;
        const int nst = (U.t1 - U.t0 + STAGE_TOK - 1) / STAGE_TOK;
        for (int s = 0; s < nst; ++s, ++sg) {
            const int buf = sg % NSTAGE;
            ok = consumer_stage_wait(&S.full[buf], (sg / NSTAGE) & 1, P.err, KVQ_SPIN_LIMIT, ok, &S.abort_flag);
            const int r0 = U.t0 + s * STAGE_TOK + 32 * warp;
            const int n = min(32, U.t1 - r0);
            if (ok && n > 0) {
                const uint8_t *kc = S.kc[buf] + 32 * warp * KVQ_D + 4 * lane;
                const uint8_t *vc = S.vc[buf] + 32 * warp * KVQ_D + 4 * lane;
                const uint16_t(*ks)[4] = S.ks[buf] + 32 * warp;
                const uint16_t(*vs)[4] = S.vs[buf] + 32 * warp;
                const int32_t *sl = S.slot[buf] + 32 * warp;
                auto kfn = [=](int tt, float kv[4]) {
                    float d[4];
                    code_minus_dither4(P, *reinterpret_cast<const uint32_t *>(kc + tt * KVQ_D), c2, 0u, sl[tt], lane, d);
                    const float sc = h2f(ks[tt][gi]);
                    kv[0] = sc * d[0];
                    kv[1] = sc * d[1];
                    kv[2] = sc * d[2];
                    kv[3] = sc * d[3];
                };
                auto vfn = [=](int tt, float vv[4]) {
                    float d[4];
                    code_minus_dither4(P, *reinterpret_cast<const uint32_t *>(vc + tt * KVQ_D), c2 | 0x10000u, 0u,
                                       sl[tt], lane, d);
                    const float sc = h2f(vs[tt][gi]);
                    vv[0] = sc * d[0];
                    vv[1] = sc * d[1];
                    vv[2] = sc * d[2];
                    vv[3] = sc * d[3];
                };
                tile<2, 8>(n, wk2, kfn, vfn, H, S.pw[warp], S.red[warp], lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[buf]);
        }
        write_unit(S, H, P.ws_o, P.ws_lse, (int64_t)U.b * P.Hq + U.kvh * g, g, P.splits, U.split, warp, lane);
    }
}

cudaError_t launch_decode_int8_token(const kvq_config *cfg, const kvq_int8_token_cache *c, const void *q,
                                     const DecodePlan &p, void *ws, cudaStream_t st) {
    ParamsT P;
    P.seq_len = c->seq_len;
    P.table = c->slot_table;
    P.k_codes = static_cast<const int8_t *>(c->k_codes);
    P.v_codes = static_cast<const int8_t *>(c->v_codes);
    P.k_scale = static_cast<const uint16_t *>(c->k_scale);
    P.v_scale = static_cast<const uint16_t *>(c->v_scale);
    P.q = static_cast<const uint16_t *>(q);
    P.ws_o = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_o);
    P.ws_lse = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + p.off_lse);
    P.err = device_error_ptr();
    P.B = c->batch;
    P.Hq = cfg->n_q_heads;
    P.Hkv = cfg->n_kv_heads;
    P.g = cfg->n_q_heads / cfg->n_kv_heads;
    P.splits = p.splits;
    P.chunk = p.chunk;
    P.cap = c->max_seq_len;
    P.n_slots = c->n_slots;
    P.nsc = KVQ_D / cfg->int8_group;
    P.gshift = cfg->int8_group == 32 ? 3 : cfg->int8_group == 64 ? 4 : 5;
    P.ctr2_layer = (uint32_t)c->layer << 17;
    const uint32_t k0 = (uint32_t)(c->seed & 0xFFFFFFFFu), k1 = (uint32_t)(c->seed >> 32);
    for (int r = 0; r < 10; ++r) {
        P.rk0[r] = k0 + (uint32_t)r * 0x9E3779B9u;
        P.rk1[r] = k1 + (uint32_t)r * 0xBB67AE85u;
    }
    P.alpha = sm_scale_of(cfg) * 1.4426950408889634f;
    if (!P.err) return cudaErrorInvalidDevicePointer;
    if (P.g > GMAX) return cudaErrorInvalidValue;
    const size_t smem = sizeof(SmemT);
    static std::atomic<uint64_t> attr_done{0};
    if (cudaError_t e = smem_opt_in(int8_token_decode_kernel, smem, attr_done)) return e;
    const int64_t n_units = (int64_t)c->batch * cfg->n_kv_heads * p.splits;
    int64_t grid = (int64_t)num_sms() * 2;
    if (grid > n_units) grid = n_units;
    int8_token_decode_kernel<<<(unsigned)grid, 32 * (NCWARP + 1), smem, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kvq
