// Device helpers shared by the kvq kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvq.h"

#define KVQ_D 128
#define KVQ_SUSPEND_NS 20000u      // mbarrier try_wait suspend hint (ns)
#define KVQ_SPIN_LIMIT (1u << 16)   // bounded mbarrier waits: about 1.3 s at most

namespace kvq {

// ---------------------------------------------------------------------------
// fp16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f2h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint16_t f2h_rd(float f) { return __half_as_ushort(__float2half_rd(f)); }
__device__ __forceinline__ uint16_t f2h_ru(float f) { return __half_as_ushort(__float2half_ru(f)); }

// d = a * b + c with f16 a, b and an f32 accumulator (one rounding, exact product).
__device__ __forceinline__ float fma_f16f32(uint16_t a, uint16_t b, float c) {
    float d;
    asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
    return d;
}
// packed fp32 pair helpers for fma.rn.f32x2 (two FMAs per instruction)
__device__ __forceinline__ unsigned long long pack2f(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ unsigned long long pack2u(uint32_t a, uint32_t b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ float lo2f(unsigned long long v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2f(unsigned long long v) { return __uint_as_float((uint32_t)(v >> 32)); }
// d = a * b + c elementwise on fp32 pairs (denormal inputs honoured: no ftz)
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint16_t lo16(uint32_t v) { return (uint16_t)(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return (uint16_t)(v >> 16); }

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3")
// ---------------------------------------------------------------------------
struct philox_key { uint32_t k0, k1; };

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
    const uint32_t MA = 0xD2511F53u, MB = 0xCD9E8D57u;
    const uint32_t WA = 0x9E3779B9u, WB = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint32_t hA = __umulhi(MA, c.x), lA = MA * c.x;
        uint32_t hB = __umulhi(MB, c.z), lB = MB * c.z;
        uint4 n;
        n.x = hB ^ c.y ^ k0;
        n.y = lB;
        n.z = hA ^ c.w ^ k1;
        n.w = lA;
        c = n;
        k0 += WA;
        k1 += WB;
    }
    return c;
}

// Dither xi in [-1/2, 1/2) from one Philox output word.
__device__ __forceinline__ float dither_from_word(uint32_t w) {
    return __fsub_rn(__uint2float_rn(w >> 8) * 0x1.0p-24f, 0.5f);
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk async copy (TMA engine, no tensor map)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
// try_wait with a suspend-time hint: the thread sleeps (up to the hint, in ns)
// until the phase completes instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(KVQ_SUSPEND_NS) : "memory");
    return ok != 0;
}
// Bounded wait (at most about limit * KVQ_SUSPEND_NS): false, and the
// device error flag set, if the phase never completes.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err,
                                          uint32_t limit = KVQ_SPIN_LIMIT) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicOr(err, 1u);
    return false;
}
// ---------------------------------------------------------------------------
// The stage ring of the decode kernels: a producer fills slots with bulk
// copies that complete on the slot's full barrier; consumer warps wait on it,
// read the slot, then arrive on its empty barrier; the producer refills a slot
// once its empty barrier completes.  A full barrier may be armed again only
// after its armed phase has completed (a second arrive on one phase is not
// allowed), and the consumers' successful waits are what guarantee that.  So
// a consumer warp whose bounded wait gives up raises the ring's abort flag
// before its next arrive on an empty barrier, the producer reads the flag
// after each of its empty waits and stops filling, and before the CTA exits
// the producer waits (bounded) for the last phase it armed on every slot, so
// that no copy is in flight.
// ---------------------------------------------------------------------------
// Consumer side: the warp's bounded wait for a stage; false for the whole warp
// if any lane gave up (the flag then raised), and false without waiting once
// the warp has failed before.
__device__ __forceinline__ bool consumer_stage_wait(uint64_t *full, uint32_t parity, unsigned *err, uint32_t limit,
                                                    bool ok, int *abort_flag) {
    if (!ok) return false;
    const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(full, parity, err, limit));
    if (!got) *reinterpret_cast<volatile int *>(abort_flag) = 1;
    return got;
}
// Producer side: raised by a consumer (read after an empty wait, whose acquire
// orders it after the consumer's flag store and arrive).
__device__ __forceinline__ bool ring_aborted(const int *abort_flag) {
    return *reinterpret_cast<const volatile int *>(abort_flag) != 0;
}
// Producer side: wait for the last armed phase of every slot (armed[j] phases
// were armed on slot j).
template <int NST>
__device__ __forceinline__ void producer_drain(uint64_t *full, const int (&armed)[NST], unsigned *err,
                                               uint32_t limit = KVQ_SPIN_LIMIT) {
#pragma unroll
    for (int j = 0; j < NST; ++j)
        if (armed[j] > 0) mbar_wait(&full[j], (uint32_t)(armed[j] - 1) & 1u, err, limit);
}

// Global -> shared bulk copy completing on `bar`; src, dst 16-B aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// Value accumulation of one token's 32 channels (one lane's block) in exact
// fp32 products.  The token's 8 bytes (32 2-bit codes, channel 4b+i of byte b
// at bits 2i) are split into 16-bit halves so that every code sits below the
// fp32 exponent field; masked in place and read as an fp32 bit pattern a code
// is the denormal code * 2^(k-149) (k = 2i, or 8 + 2i for odd bytes).  One
// weight pair ps * (2^(149-EV), 2^(141-EV)) serves every bit position, so a
// packed fma.rn.f32x2 adds code * ps * 2^(2i-EV): accumulator i carries an
// extra 2^(2i), removed once per unit by value_block_reduce.
// acc2[8*wi + 4*ab + i] holds channels (16 wi + 8 ab + i, 16 wi + 8 ab + 4 + i)
// of the block.  |p s| < 2^16 keeps the weights below 2^127.
// ---------------------------------------------------------------------------
#define KVQ_EV 38
__device__ __forceinline__ void value_token_accum(uint2 codes, float ps, unsigned long long acc2[16]) {
    const unsigned long long wt = pack2f(ps * __int_as_float((127 + 149 - KVQ_EV) << 23),
                                         ps * __int_as_float((127 + 141 - KVQ_EV) << 23));
    const uint32_t uw[2] = {codes.x, codes.y};
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
        const uint32_t w0 = uw[wi], w16 = uw[wi] >> 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t m0 = 3u << (2 * i), m1 = 3u << (8 + 2 * i);
            acc2[8 * wi + i] = ffma2(pack2u(w0 & m0, w0 & m1), wt, acc2[8 * wi + i]);
            acc2[8 * wi + 4 + i] = ffma2(pack2u(w16 & m0, w16 & m1), wt, acc2[8 * wi + 4 + i]);
        }
    }
}

// The 4-bit form: the token's 16 bytes (32 4-bit codes, channel 2b + i of
// byte b at bits 4i).  Halves of each word are masked the same way; channel
// 2b + i carries an extra 2^(4i), and acc2[4*wi + 2*ab + i] holds channels
// (8 wi + 4 ab + i, 8 wi + 4 ab + 2 + i).  Codes stay below bit 16, so every
// masked word is still a denormal and every product exact.
__device__ __forceinline__ void value_token_accum4(uint4 codes, float ps, unsigned long long acc2[16]) {
    const unsigned long long wt = pack2f(ps * __int_as_float((127 + 149 - KVQ_EV) << 23),
                                         ps * __int_as_float((127 + 141 - KVQ_EV) << 23));
    const uint32_t uw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t w0 = uw[wi], w16 = uw[wi] >> 16;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t m0 = 15u << (4 * i), m1 = 15u << (8 + 4 * i);
            acc2[4 * wi + i] = ffma2(pack2u(w0 & m0, w0 & m1), wt, acc2[4 * wi + i]);
            acc2[4 * wi + 2 + i] = ffma2(pack2u(w16 & m0, w16 & m1), wt, acc2[4 * wi + 2 + i]);
        }
    }
}

// Packed fp32 add, and a 64-bit register pair exchanged across lanes.
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long shfl_xor2(unsigned long long v, int o) {
    return pack2f(__shfl_xor_sync(0xFFFFFFFFu, lo2f(v), o), __shfl_xor_sync(0xFFFFFFFFu, hi2f(v), o));
}

// The value accumulators summed over the eight lanes of a channel block (lanes 4ts + jg, ts = 0..7),
// with the result scattered: lane ts keeps channels 4ts .. 4ts + 3 of the block, scaled back by their
// bit-position powers.  At 2 bits channel 4ts + i is half ts % 2 of acc2[8 (ts / 4) + 4 ((ts / 2) % 2) + i]
// carrying 2^(2i - EV); at 4 bits channel 4ts + x is acc2[2ts + (x & 1)], low half for x < 2, carrying
// 2^(4 (x & 1) - EV).  Three exchange levels over the lane bits 4, 3, 2 (ts bits 2, 1, 0), each keeping
// the half of the remaining floats that the lane's side owns: pairs 8b .. 8b + 7 (b = ts bit 2), then four
// of them (ts bit 1), then one half of each of the four pairs (2 bits) or two of the pairs (4 bits).
template <int BV>
__device__ __forceinline__ float4 value_block_reduce(const unsigned long long acc2[16], int ts) {
    const bool b2 = (ts & 4) != 0, b1 = (ts & 2) != 0, b0 = (ts & 1) != 0;
    unsigned long long a8[8], a4[4];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        a8[k] = add2(b2 ? acc2[8 + k] : acc2[k], shfl_xor2(b2 ? acc2[k] : acc2[8 + k], 16));
#pragma unroll
    for (int k = 0; k < 4; ++k) a4[k] = add2(b1 ? a8[4 + k] : a8[k], shfl_xor2(b1 ? a8[k] : a8[4 + k], 8));
    if (BV == 2) {
        float f[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            f[k] = (b0 ? hi2f(a4[k]) : lo2f(a4[k])) + __shfl_xor_sync(0xFFFFFFFFu, b0 ? lo2f(a4[k]) : hi2f(a4[k]), 4);
        return make_float4(f[0] * __int_as_float((127 + KVQ_EV) << 23), f[1] * __int_as_float((127 + KVQ_EV - 2) << 23),
                           f[2] * __int_as_float((127 + KVQ_EV - 4) << 23), f[3] * __int_as_float((127 + KVQ_EV - 6) << 23));
    } else {
        unsigned long long a2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) a2[k] = add2(b0 ? a4[2 + k] : a4[k], shfl_xor2(b0 ? a4[k] : a4[2 + k], 4));
        return make_float4(lo2f(a2[0]) * __int_as_float((127 + KVQ_EV) << 23),
                           lo2f(a2[1]) * __int_as_float((127 + KVQ_EV - 4) << 23),
                           hi2f(a2[0]) * __int_as_float((127 + KVQ_EV) << 23),
                           hi2f(a2[1]) * __int_as_float((127 + KVQ_EV - 4) << 23));
    }
}

__device__ __forceinline__ void scale_pairs(unsigned long long acc2[16], float sc) {
    const unsigned long long s2 = pack2f(sc, sc);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        unsigned long long d;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(acc2[i]), "l"(s2));
        acc2[i] = d;
    }
}

// A cached length as the decode kernels use it: seq_len[b] clamped into
// [0, max_len], so that a corrupt length can never move a read outside the
// caller's arrays; a clamped length records KVQ_DEVICE_ERR_CAPACITY.
__device__ __forceinline__ int clamp_len(int L, int max_len, unsigned *err) {
    if (L < 0 || L > max_len) {
        atomicOr(err, KVQ_DEVICE_ERR_CAPACITY);
        L = L < 0 ? 0 : max_len;
    }
    return L;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace kvq
