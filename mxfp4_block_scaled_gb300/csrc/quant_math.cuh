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

// |bf16| pair maxima: the sign-cleared bit patterns of non-NaN bf16 values
// order like their magnitudes, so a 16-bit unsigned max is an exact abs-max.
__device__ __forceinline__ uint32_t absmax8(const uint4& v, uint32_t m) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
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

// NVFP4 scale byte of a block with abs-max amax_b under global scale sg.
__device__ __forceinline__ uint32_t nvfp4_scale_byte(float amax_b, float sg) {
    const float p = __fmul_rn(sg, 6.0f);
    return p > 0.0f ? cvt_e4m3(__fdiv_rn(amax_b, p)) : 0u;
}

// NVFP4 codes of 8 elements of a block with scale byte sbyte under sg.
__device__ __forceinline__ uint32_t nvfp4_codes8(const uint4& v, uint32_t sbyte, float sg) {
    const float d = __fmul_rn(e4m3_to_f32(sbyte), sg);
    if (d == 0.0f) return 0u;
    float f[8];
    unpack8(v, f);
    if (d >= 1.1754944e-38f && d <= 8.5070592e37f) return e2m1_word(f, d, __frcp_rn(d));
    return e2m1_word_exact(f, d);
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
