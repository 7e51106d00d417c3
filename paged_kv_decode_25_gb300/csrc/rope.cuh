// Exact RoPE rotation of one bf16 pair element: RN_bf16(RN_f64(a*b + c*d))
// for bf16 a, c and fp32 table values b, d (each product exact in double),
// computed in single precision when that provably gives the same bits, else
// in double. Shared by the append kernel and the fused decode step, so both
// write the same bits.
#pragma once

#include "common.cuh"

namespace mi {

// Exact widening to double built from the bit fields (integer work only);
// zero, subnormal, infinite and NaN inputs take the hardware conversion.
__device__ __forceinline__ double bf16_bits_to_f64(uint32_t h) {
    const uint32_t e = (h >> 7) & 0xFFu;
    if (e == 0u || e == 0xFFu) return (double)__uint_as_float(h << 16);
    const uint32_t hi = ((h & 0x8000u) << 16) | ((e + 896u) << 20) | ((h & 0x7Fu) << 13);
    return __hiloint2double((int)hi, 0);
}

__device__ __forceinline__ double f32_to_f64_bits(float f) {
    const uint32_t u = __float_as_uint(f);
    const uint32_t e = (u >> 23) & 0xFFu;
    if (e == 0u || e == 0xFFu) return (double)f;
    const uint32_t m = u & 0x7FFFFFu;
    const uint32_t hi = (u & 0x80000000u) | ((e + 896u) << 20) | (m >> 3);
    return __hiloint2double((int)hi, (int)(m << 29));
}

// y = RN_bf16(RN_double(a*b - c*d)) with every product exact in double: the
// fma forms a*b - (c*d) exactly and rounds once, as the two-step form does.
__device__ __forceinline__ uint32_t rot_lo(double a, double b, double c, double d) {
    return f64_to_bf16(fma(a, b, -(c * d)));
}
__device__ __forceinline__ uint32_t rot_hi(double a, double b, double c, double d) {
    return f64_to_bf16(fma(a, b, c * d));
}

// RN_bf16(RN_double(a*b + c*d)) for bf16 a, c and fp32 b, d, in single
// precision when that decides it. q = RN(c*d) and its rounding error qe (an
// fma recovers it exactly above the underflow range) give c*d = q + qe; the
// fma s = RN(a*b + q) rounds the exact a*b + q once, so
//   |exact - s| <= |qe| + ulp(s)/2 <= |qe| + |s| 2^-24 <= err,
// err being that sum (plus 2^-140 for a product c*d that underflowed)
// rounded upward. lo = s - err rounded down and hi = s + err rounded up
// enclose the exact value and its double rounding; rounding to bf16 is
// monotone, so when lo and hi round to the same bf16 the exact value does
// too, and so does s. Returns s and sets lo and hi; the caller rounds pairs
// of values, and of their lo and hi, with the hardware conversion and
// compares the packed ends a pair at a time. `slow` is set here when s is
// zero, tiny (below 2^-100), huge or not finite, or q tiny but not zero;
// the caller then (or when the ends differ) takes the double-precision
// route. The _rn intrinsics keep the compiler from contracting c*d into an
// fma, which would break the split. (An earlier test on the bit patterns,
// about twenty integer operations per value, made the prefill append
// ALU-bound.)
__device__ __forceinline__ float rot_fast(float a, float b, float c, float d, float& lo, float& hi, bool& slow) {
    const float q = __fmul_rn(c, d);
    const float qe = fmaf(c, d, -q);
    const float s = fmaf(a, b, q);
    const float as = fabsf(s);
    const float err = __fmaf_ru(as, 0x1p-24f, __fadd_ru(fabsf(qe), 0x1p-140f));
    lo = __fsub_rd(s, err);
    hi = __fadd_ru(s, err);
    slow |= !(as >= 0x1p-100f && as < 0x1p127f && (fabsf(q) >= 0x1p-100f || q == 0.f));
    return s;
}

// The double-precision route of a rotated word: the exact products and one
// double rounding decide the bits. Out of line and called only from a
// separate pass after a caller's rotation loop (rotate_word_fast flags the
// words that need it): a call site inside the loop, even untaken, cost ~650
// cycles per word, and the route inlined there made the code several times
// larger.
static __device__ __noinline__ uint2 rotate_word_exact(uint32_t xl, uint32_t xh, float4 cs) {
    const double a0 = bf16_bits_to_f64(xl & 0xFFFFu), a1 = bf16_bits_to_f64(xl >> 16);
    const double b0 = bf16_bits_to_f64(xh & 0xFFFFu), b1 = bf16_bits_to_f64(xh >> 16);
    const double c0 = f32_to_f64_bits(cs.x), sn0 = f32_to_f64_bits(cs.y);
    const double c1 = f32_to_f64_bits(cs.z), sn1 = f32_to_f64_bits(cs.w);
    return make_uint2(rot_lo(a0, c0, b0, sn0) | (rot_lo(a1, c1, b1, sn1) << 16),
                      rot_hi(b0, c0, a0, sn0) | (rot_hi(b1, c1, a1, sn1) << 16));
}

// Rotated bf16 pairs of one group: element k of the first half (lo) and of
// the second half (hi) of a head, two adjacent pairs per word:
// ylo = x_lo * cos - x_hi * sin, yhi = x_hi * cos + x_lo * sin,
// cs = (cos, sin) of pair 2j and (cos, sin) of pair 2j + 1.
// Single precision only; returns true when one of the four values needs
// the exact route, in which case the caller replaces (yl, yh) by
// rotate_word_exact(xl, xh, cs).
__device__ __forceinline__ bool rotate_word_fast(uint32_t xl, uint32_t xh, float4 cs, uint32_t& yl,
                                                 uint32_t& yh) {
    const float fa0 = bf16_lo(xl), fa1 = bf16_hi(xl);
    const float fb0 = bf16_lo(xh), fb1 = bf16_hi(xh);
    bool slow = false;
    float lo0, hi0, lo1, hi1, lo2, hi2, lo3, hi3;
    const float s0 = rot_fast(fa0, cs.x, -fb0, cs.y, lo0, hi0, slow);
    const float s1 = rot_fast(fa1, cs.z, -fb1, cs.w, lo1, hi1, slow);
    const float s2 = rot_fast(fb0, cs.x, fa0, cs.y, lo2, hi2, slow);
    const float s3 = rot_fast(fb1, cs.z, fa1, cs.w, lo3, hi3, slow);
    yl = pack_bf16x2(s0, s1);
    yh = pack_bf16x2(s2, s3);
    // both ends of each value's interval round alike: a pair at a time
    slow |= pack_bf16x2(lo0, lo1) != pack_bf16x2(hi0, hi1) || pack_bf16x2(lo2, lo3) != pack_bf16x2(hi2, hi3);
    return slow;
}

}  // namespace mi
