// Write-side helpers of the quantization kernels (sm_103a): the asymmetric
// min-max fit and the code of an element, and the INT8 dithered code.  Only
// the write side includes this header.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

// Asymmetric min-max fit for b-bit codes (same rules as the C ABI states):
//   z = fp16 round-down(mn); s = fp16 round-up(fp32 (mx - z) / qmax), raised
//   one fp16 step while z + qmax*s < mx (an exact test);
//   s = 0 when mx == mn.
// mn and mx are fp16 values.  The test is exact in fp32: p = qmax*s has at
// most 15 significant bits (an fp16 s times qmax <= 15), so p is an fp32
// number, and for an fp32 p, p < mx - z holds exactly iff p < fl_up(mx - z)
// (fl_up(mx - z) is the least fp32 number >= mx - z; when mx - z is not an
// fp32 number no fp32 number lies strictly between it and fl_up).
__device__ __forceinline__ void affine_fit(float mn, float mx, int qmax, uint16_t &s, uint16_t &z) {
    z = f2h_rd(mn);
    s = 0;
    if (mx > mn) {
        float zf = h2f(z);
        float range = __fsub_rn(mx, zf);
        float s32 = __fdiv_rn(range, (float)qmax);
        s = f2h_ru(s32);
        const float up = __fsub_ru(mx, zf);
        while (__fmul_rn(h2f(s), (float)qmax) < up) s = (uint16_t)(s + 1);
    }
}

// code = clamp(rint((x - z) / s), 0, qmax) with the quotient rounded to
// nearest in fp32 (the definition); 0 when s == 0.  rinv = fl(1 / s).  The
// product d * rinv differs from fl(d / s) by at most 2^-17 when |d / s| <= 32
// (three roundings of 2^-24 relative), so its nearest integer is the
// quotient's unless it lies within 2^-16.6 of a half-integer; only then is
// the quotient itself formed.
__device__ __forceinline__ int affine_code(float x, float zf, float sf, float rinv, int qmax) {
    if (sf == 0.0f) return 0;
    const float d = __fsub_rn(x, zf);
    const float qa = __fmul_rn(d, rinv);
    float r = rintf(qa);
    if (fabsf(__fsub_rn(qa, r)) > 0.49999f) r = rintf(__fdiv_rn(d, sf));
    r = fminf(fmaxf(r, 0.0f), (float)qmax);
    return (int)r;
}

// The code of an element of a group fitted by affine_fit, without the
// quotient: rint(d * rinv).  For x in [mn, mx], d = fl(x - z) lies in
// [0, qmax*s] (z <= mn, and qmax*s is an fp32 number >= mx - z), so the
// result lies in [0, qmax] and needs no clamp; with s = 0 (rinv = 0, every
// x = z) it is 0.  `tie` is set when the product lies within 2^-16.6 of a
// half-integer, where only affine_code's quotient decides: callers then
// recompute that element (or their whole set) with affine_code.
__device__ __forceinline__ int affine_code_fast(float x, float zf, float rinv, bool &tie) {
    const float qa = __fmul_rn(__fsub_rn(x, zf), rinv);
    const float r = rintf(qa);
    tie |= fabsf(__fsub_rn(qa, r)) > 0.49999f;
    return (int)r;
}

// INT8 dithered code = clamp(rint(fl(x / s) + xi), -127, 127) in fp32 with
// rounding to nearest (the definition), s != 0, rinv = fl(1 / s).  With
// |x / s| < 127 the product x * rinv is within 2^-15.4 of fl(x / s), so the
// sums with xi differ by at most 2^-15 and round to the same integer unless
// they lie within 2^-13.3 of a half-integer; only then is the quotient formed.
__device__ __forceinline__ int dither_code(float x, float s, float rinv, float xi) {
    const float va = __fadd_rn(__fmul_rn(x, rinv), xi);
    float r = rintf(va);
    if (fabsf(__fsub_rn(va, r)) > 0.4999f) r = rintf(__fadd_rn(__fdiv_rn(x, s), xi));
    return (int)fminf(fmaxf(r, -127.f), 127.f);
}

}  // namespace kvq
