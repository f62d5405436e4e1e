// quant_math.cuh -- the per-block arithmetic of the NVFP4 / MXFP4 quantisers,
// shared by the quantise kernels and the fused decode GEMM (one definition,
// so both produce the same bits).
//
// NVFP4 ("vLLM on DGX Spark: technical report", section 6.1 "NVFP4 format"):
// per 16-element K block, s_b = E4M3_rne_satfinite(amax_b / fl(6 s_g)),
// d = fl(s_b * s_g), element = E2M1_rne_satfinite(fl(x / d)), 0 when d == 0.
// MXFP4 (same page, section 6.4): per 32-element block, E8M0 exponent
// e = floor(log2 amax_b) - 2 (clamped to [-127, 127]); element =
// E2M1_rne_satfinite(x * 2^-e) (exact), all-zero blocks give byte 0 and zeros.
#pragma once

#include "common.cuh"

namespace fp4 {

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// |bf16| pair maxima: the sign-cleared bit patterns of non-NaN bf16 values
// order like their magnitudes, so a 16-bit unsigned max is an exact abs-max.
__device__ __forceinline__ uint32_t absmax8(const uint4& v, uint32_t m) {
    m = max_u16x2(m, v.x & 0x7FFF7FFFu);
    m = max_u16x2(m, v.y & 0x7FFF7FFFu);
    m = max_u16x2(m, v.z & 0x7FFF7FFFu);
    m = max_u16x2(m, v.w & 0x7FFF7FFFu);
    return m;
}

// E2M1 codes of x / d for 8 elements (one 32-bit word), bit-identical to
// converting the correctly rounded quotients fl(x / d).  With rd = fl(1/d),
// q = fl(x * rd) is within 1.5 * 2^-23 relative of x / d, and so is fl(x / d);
// q * (1 - 2^-21) and q * (1 + 2^-21) (each rounded) therefore bracket
// fl(x / d).  E2M1 rounding is monotone, so when both brackets give the same
// codes those are the codes of fl(x / d).  Otherwise (a quotient next to a
// rounding threshold, rare) the codes come from correctly rounded divisions.
// d must be a normal float whose reciprocal is normal.
__device__ __forceinline__ uint32_t e2m1_word(const float* f, float d, float rd) {
    const float lo_s = 1.0f - 4.76837158203125e-07f;  // 1 - 2^-21
    const float hi_s = 1.0f + 4.76837158203125e-07f;  // 1 + 2^-21
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(f[i], rd);
    const uint32_t lo = cvt_e2m1x8(__fmul_rn(q[0], lo_s), __fmul_rn(q[1], lo_s), __fmul_rn(q[2], lo_s),
                                   __fmul_rn(q[3], lo_s), __fmul_rn(q[4], lo_s), __fmul_rn(q[5], lo_s),
                                   __fmul_rn(q[6], lo_s), __fmul_rn(q[7], lo_s));
    const uint32_t hi = cvt_e2m1x8(__fmul_rn(q[0], hi_s), __fmul_rn(q[1], hi_s), __fmul_rn(q[2], hi_s),
                                   __fmul_rn(q[3], hi_s), __fmul_rn(q[4], hi_s), __fmul_rn(q[5], hi_s),
                                   __fmul_rn(q[6], hi_s), __fmul_rn(q[7], hi_s));
    if (lo == hi) return lo;
    return cvt_e2m1x8(__fdiv_rn(f[0], d), __fdiv_rn(f[1], d), __fdiv_rn(f[2], d), __fdiv_rn(f[3], d),
                      __fdiv_rn(f[4], d), __fdiv_rn(f[5], d), __fdiv_rn(f[6], d), __fdiv_rn(f[7], d));
}

__device__ __forceinline__ uint32_t e2m1_word_exact(const float* f, float d) {
    return cvt_e2m1x8(__fdiv_rn(f[0], d), __fdiv_rn(f[1], d), __fdiv_rn(f[2], d), __fdiv_rn(f[3], d),
                      __fdiv_rn(f[4], d), __fdiv_rn(f[5], d), __fdiv_rn(f[6], d), __fdiv_rn(f[7], d));
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    f[0] = bf16lo(v.x), f[1] = bf16hi(v.x), f[2] = bf16lo(v.y), f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z), f[5] = bf16hi(v.z), f[6] = bf16lo(v.w), f[7] = bf16hi(v.w);
}

// E4M3 byte of fl(a / p) (round to nearest even, saturating) from the product
// t = fl(a * fl(1/p)): t is within 1.5 * 2^-23 relative of fl(a / p) when p and
// 1/p are normal floats, so t * (1 -/+ 2^-21) bracket it and, E4M3 rounding
// being monotone, equal conversions of the brackets are the conversion of
// fl(a / p).  Otherwise (a quotient next to a rounding threshold) the byte
// comes from the correctly rounded division.
__device__ __forceinline__ uint32_t e4m3_of_quotient(float a, float p, float inv_p) {
    const float t = __fmul_rn(a, inv_p);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(r)
        : "f"(__fmul_rn(t, 1.0f + 4.76837158203125e-07f)), "f"(__fmul_rn(t, 1.0f - 4.76837158203125e-07f)));
    const uint32_t lo = r & 0xFFu, hi = (uint32_t)r >> 8;
    if (lo == hi) return lo;
    return cvt_e4m3(__fdiv_rn(a, p));
}

// 1/p for the bracketed NVFP4 scale byte (p = fl(6 s_g)): fl(1/p) when p and
// 1/p are normal floats with room for the bracket, else 0 (division path).
__device__ __forceinline__ float nvfp4_inv_p(float p) {
    return (p >= 2.3509887e-38f && p <= 4.2535296e37f) ? __frcp_rn(p) : 0.0f;
}

// NVFP4 scale byte E4M3(fl(amax_b / p)) of a block; 0 when p is not positive.
// amax_b >= 0, so the byte is below 0x80.
__device__ __forceinline__ uint32_t nvfp4_scale_byte(float amax_b, float p, float inv_p) {
    if (inv_p != 0.0f) return e4m3_of_quotient(amax_b, p, inv_p);
    return p > 0.0f ? cvt_e4m3(__fdiv_rn(amax_b, p)) : 0u;
}

// A multiplier r for which E2M1(fl(x * r)) equals E2M1(fl(x / d)) for every
// bf16 x, or 0 when none is proven; 2^-120 <= d <= 2^120, rd = fl(1/d).
//
// E2M1 round-to-nearest-even with saturation depends only on where a value
// lies against the midpoints m in {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5},
// whose significands are 1, 1.25, 1.5 and 1.75.  For r within 1.5 ulp of
// 1/d, fl(x / d) and fl(x * r) are both within 2^-21 relative of x / d
// (values too small for a normal float give a zero code on both sides; too
// large ones saturate on both).  So for an x farther than 2^-19 m d from m d,
// x / d is farther than 2^-19 m from m, both results lie strictly on its side
// of m, and they agree there.  The distance runs on integer significands:
// with md the 24-bit significand of d, m d has the significand md * s
// (s = 4..7, m's significand times 4); in the binade of that product
// (leading bit L) the bf16 values are the multiples of 2^(L-7), and a
// distance above 2^(L-18) to the nearest bounds the relative distance below
// by 2^-19.  When every midpoint passes, r = rd.  When one fails, exactly one
// bf16 value x* lies that close (the next is about 2^-8 away); with `refine`
// the candidates rd, rd + 1 ulp and rd - 1 ulp are tried, and one is taken
// when, for each failing midpoint, the code of fl(x* * r) equals the code of
// fl(x* / d) (and so, by symmetry, for -x*).
__device__ __forceinline__ bool e2m1_class_far(uint32_t md, uint32_t s) {
    const uint32_t p = md * s;  // < 2^27
    const int L = 31 - __clz((int)p);
    const uint32_t g = 1u << (L - 7);
    const uint32_t r = p & (g - 1u);
    return min(r, g - r) > (1u << (L - 18));
}

__device__ __forceinline__ float round_to_bf16(float v) {  // finite v
    uint32_t u = __float_as_uint(v);
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    return __uint_as_float(u);
}

__device__ __forceinline__ float e2m1_product_multiplier(float d, float rd, bool refine) {
    if (!(d >= 7.5231638e-37f && d <= 1.3292280e36f)) return 0.0f;  // 2^-120, 2^120
    const uint32_t md = (__float_as_uint(d) & 0x7FFFFFu) | 0x800000u;
    const bool far4 = e2m1_class_far(md, 4), far5 = e2m1_class_far(md, 5);
    const bool far6 = e2m1_class_far(md, 6), far7 = e2m1_class_far(md, 7);
    if (far4 && far5 && far6 && far7) return rd;
    if (!refine) return 0.0f;
    const float mids[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
    const bool far[7] = {far4, far6, far5, far7, far5, far7, far5};
    for (int c = 0; c < 3; ++c) {
        const float r = __uint_as_float(__float_as_uint(rd) + (c == 0 ? 0u : c == 1 ? 1u : 0xFFFFFFFFu));
        bool ok = true;
#pragma unroll
        for (int i = 0; i < 7; ++i) {
            if (far[i]) continue;
            const float xs = round_to_bf16(__fmul_rn(mids[i], d));
            ok = ok && cvt_e2m1x2(__fdiv_rn(xs, d), 0.0f) == cvt_e2m1x2(__fmul_rn(xs, r), 0.0f);
        }
        if (ok) return r;
    }
    return 0.0f;
}

// The divisor of NVFP4 scale byte `sbyte` under global scale sg, as used by
// nvfp4_word: x = d = fl(E4M3(sbyte) * sg); y = the multiplier of the
// product path (e2m1_product_multiplier) when one is proven for every bf16
// input, -fl(1/d) when only the bracket of e2m1_word applies, 0 when d or 1/d
// is not a normal float (correctly rounded divisions; also d == 0, where
// every code is 0).
__device__ __forceinline__ float2 nvfp4_divisor(uint32_t sbyte, float sg, bool refine) {
    const float d = __fmul_rn(e4m3_to_f32(sbyte), sg);
    if (!(d >= 1.1754944e-38f && d <= 8.5070592e37f)) return make_float2(d, 0.0f);
    const float rd = __frcp_rn(d);
    const float r = e2m1_product_multiplier(d, rd, refine);
    return make_float2(d, r != 0.0f ? r : -rd);
}

// NVFP4 codes of 8 elements (one 32-bit word) with the divisor entry e of
// their block; 0 when d == 0.
__device__ __forceinline__ uint32_t nvfp4_word(const float* f, float2 e) {
    if (e.y > 0.0f)
        return cvt_e2m1x8(__fmul_rn(f[0], e.y), __fmul_rn(f[1], e.y), __fmul_rn(f[2], e.y), __fmul_rn(f[3], e.y),
                          __fmul_rn(f[4], e.y), __fmul_rn(f[5], e.y), __fmul_rn(f[6], e.y), __fmul_rn(f[7], e.y));
    if (e.x == 0.0f) return 0u;
    if (e.y < 0.0f) return e2m1_word(f, e.x, -e.y);
    return e2m1_word_exact(f, e.x);
}

// MXFP4 scale byte (E8M0, 0 for an all-zero block) and the factor 2^-e.
__device__ __forceinline__ uint32_t mxfp4_scale_byte(float amax_b, float& inv) {
    inv = 0.0f;
    if (!(amax_b > 0.0f)) return 0u;
    const uint32_t u = __float_as_uint(amax_b);
    const int fl = (u >> 23) ? (int)(u >> 23) - 127 : (31 - __clz((int)u)) - 149;
    int e = fl - 2;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, a normal float here
    return (uint32_t)(e + 127);
}

// MXFP4 codes of 8 elements (exact products with 2^-e).
__device__ __forceinline__ uint32_t mxfp4_codes8(const uint4& v, float inv) {
    if (inv == 0.0f) return 0u;
    float f[8];
    unpack8(v, f);
    return cvt_e2m1x8(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv), __fmul_rn(f[3], inv),
                      __fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv), __fmul_rn(f[7], inv));
}

}  // namespace fp4
