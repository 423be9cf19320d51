// Tensor-core helpers of the grouped-query decode kernels (sm_103a):
// mma.sync m16n8k16 with fp16 operands and fp32 accumulation, exact fp16
// operands made from packed 2-bit codes, and fp16 hi / lo splits of fp32
// products for the B operand.
#pragma once

#include "kvq_device.cuh"

namespace kvq {
namespace {

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// both 16-bit halves of v: lo -> e4m3x2 -> f16x2, hi -> e4m3x2 -> f16x2
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t v, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(v));
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hneg2(uint32_t a) {
    uint32_t d;
    asm("neg.f16x2 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
// ldmatrix of four 8 x 8 matrices of 16-bit elements, transposed: lanes 8m .. 8m + 7 give the
// 16-byte row addresses of matrix m; lane 4q + r receives in d[m] the elements (rows 2r, 2r + 1;
// column q) of matrix m, row 2r in the low half.  Volatile with a memory clobber: it reads
// bytes that a bulk copy wrote, so it stays behind the barrier wait that announced them.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t d[4], const void *row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(smem_addr(row))
                 : "memory");
}

// fp16x2 product a*b as its hi part (x == 0) or its lo part (x == 1):
// hi = fl(ah b); lo = fl(al b + fl(ah b - hi)), the inner FMA being exact.
// The negation is a floating-point one, which the FMA can take as an
// operand modifier.
__device__ __forceinline__ uint32_t split_prod(uint32_t ah, uint32_t al, uint32_t b, bool x) {
    uint32_t d = hmul2(ah, b);
    if (x) d = hfma2(al, b, hfma2(ah, b, hneg2(d)));
    return d;
}
// fp32 pair -> fp16x2 hi (x == 0) or lo = fl(v - hi) (x == 1); first value in the low half
__device__ __forceinline__ uint32_t split_pair(float v0, float v1, bool x) {
    uint32_t hi;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(v1), "f"(v0));
    if (!x) return hi;
    const float r0 = v0 - h2f(lo16(hi)), r1 = v1 - h2f(hi16(hi));
    uint32_t lo;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(r1), "f"(r0));
    return lo;
}

// 2^x, approximate, with results below 2^-126 flushed to zero (softmax weights that small add nothing)
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// four accumulators times sc, as two packed fp32 multiplies
__device__ __forceinline__ void scale4(float d[4], float sc) {
    const unsigned long long s2 = pack2f(sc, sc);
    unsigned long long a = pack2f(d[0], d[1]), b = pack2f(d[2], d[3]);
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(s2));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(b) : "l"(s2));
    d[0] = lo2f(a); d[1] = hi2f(a); d[2] = lo2f(b); d[3] = hi2f(b);
}

template <int N>
__device__ __forceinline__ void load_row(const uint32_t *p, uint32_t (&v)[N]) {
    if constexpr (N == 4) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    } else if constexpr (N == 2) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        v[0] = u.x; v[1] = u.y;
    } else {
        v[0] = *p;
    }
}

}  // namespace
}  // namespace kvq
