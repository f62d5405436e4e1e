// mxfp8.cu -- MXFP8 / MXFP6 quantisers: E4M3, E5M2, E2M3 or E3M2 elements in
// 32-element blocks with one E8M0 scale.  "vLLM per-format kernel capability
// matrix" lists MXFP6 and MXFP8 with group size 32; the scale rule is the
// MXFP4 one ("vLLM on DGX Spark: technical report", section 6.4) with the
// element's own largest exponent emax (E4M3 8, E5M2 15, E2M3 2, E3M2 4) in
// place of E2M1's:
//   e = floor(log2 amax_b) - emax, clamped to [-127, 127], stored as the E8M0
//   byte e + 127; element codes ELEM_rne_satfinite(x * 2^-e), one byte each
//   (the 6-bit codes in the low six bits, the top two bits zero); an
//   all-zero block gets scale byte 0 and code 0.
// x * 2^-e is exact: 2^-e is a normal float, |x| * 2^-e < 2^(emax + 1), and a
// product small enough to lose bits in fp32 lies far below every format's
// smallest step and rounds to zero either way (keeping its sign), so the
// hardware conversion rounds the exact quotient.
//
// One thread per 32-element block: four 16-byte loads, a 16-bit abs-max
// over the sign-cleared bf16 patterns, sixteen paired conversions and two
// 16-byte stores; consecutive threads take consecutive blocks of a row.
// Scale-layout padding (rows to 128, K to 256 elements) is written as 0.
#include <cuda_bf16.h>

#include "common.cuh"
#include "mxfp8.h"
#include "quant_math.cuh"

namespace fp4 {

constexpr int kMx8Threads = 256;

// Two fp32 -> two codes in 16 bits, `even` in the low byte, round to nearest
// even, saturating at the format's largest finite value.
template <int ELEM>
__device__ __forceinline__ uint32_t cvt_mx_x2(float even, float odd) {
    uint16_t r;
    if constexpr (ELEM == MX_ELEM_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(odd), "f"(even));
    else if constexpr (ELEM == MX_ELEM_E5M2)
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(odd), "f"(even));
    else if constexpr (ELEM == MX_ELEM_E2M3)
        asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(odd), "f"(even));
    else
        asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(odd), "f"(even));
    return r;
}

// The E4M3 code of the same value as a 6-bit code (E2M3 or E3M2; the low six
// bits of the byte): every E2M3 and E3M2 value is an E4M3 value (E4M3 has as
// many or more mantissa bits and a wider exponent range), so the widening is
// exact.  E2M3 (bias 1): exponent field e > 0 is 2^(e-1) (1 + m/8) -> E4M3
// field e + 6, mantissa m; e = 0 is m 2^-3 (m = 1: 2^-3; 2-3: 2^-2 (1 + (m-2)/2);
// 4-7: 2^-1 (1 + (m-4)/4)).  E3M2 (bias 3): e > 0 is 2^(e-3) (1 + m/4) -> field
// e + 4, mantissa 2m; e = 0 is m 2^-4.  Zero keeps its sign.
template <int ELEM>
__device__ __forceinline__ uint32_t fp6_to_e4m3(uint32_t c) {
    const uint32_t sign = (c & 0x20u) << 2;
    uint32_t mag;
    if constexpr (ELEM == MX_ELEM_E2M3) {
        const uint32_t e = (c >> 3) & 3u, m = c & 7u;
        if (e) {
            mag = ((e + 6u) << 3) | m;
        } else {
            // subnormal m * 2^-3: exponent of the leading bit, then the rest
            mag = m == 0u ? 0u : m == 1u ? 0x20u : m < 4u ? (0x28u | ((m & 1u) << 2)) : (0x30u | ((m & 3u) << 1));
        }
    } else {
        const uint32_t e = (c >> 2) & 7u, m = c & 3u;
        if (e) {
            mag = ((e + 4u) << 3) | (m << 1);
        } else {
            mag = m == 0u ? 0u : m == 1u ? 0x18u : m == 2u ? 0x20u : 0x24u;  // m * 2^-4
        }
    }
    return sign | mag;
}

// Four 6-bit codes (one per byte) -> four E4M3 codes.
template <int ELEM>
__device__ __forceinline__ uint32_t widen4(uint32_t w) {
    return fp6_to_e4m3<ELEM>(w & 0x3Fu) | (fp6_to_e4m3<ELEM>((w >> 8) & 0x3Fu) << 8) |
           (fp6_to_e4m3<ELEM>((w >> 16) & 0x3Fu) << 16) | (fp6_to_e4m3<ELEM>((w >> 24) & 0x3Fu) << 24);
}

template <int ELEM, bool WIDEN>
__global__ void __launch_bounds__(kMx8Threads) mx8_quant_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                                int64_t k, int64_t rows_pad, int64_t ksf,
                                                                uint8_t* __restrict__ codes,
                                                                uint8_t* __restrict__ scales) {
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    constexpr int kEmax = mx_elem_emax(ELEM);
    const int64_t kb = k / 32;  // real blocks per row
    const int64_t total = rows_pad * ksf;
    const int64_t stride = (int64_t)gridDim.x * kMx8Threads;
    for (int64_t t = (int64_t)blockIdx.x * kMx8Threads + threadIdx.x; t < total; t += stride) {
        const int64_t r = t / ksf, j = t - r * ksf;
        uint32_t sbyte = 0;
        if (r < rows && j < kb) {
            const uint4* px = reinterpret_cast<const uint4*>(x + r * k + j * 32);
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __ldg(px + i);
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) m = absmax8(v[i], m);
            m = max(m & 0xFFFFu, m >> 16);
            uint4 out[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if (m != 0) {
                const uint32_t ab = m << 16;  // fp32 bits of amax_b
                const uint32_t ef = ab >> 23;
                const int fl = ef ? (int)ef - 127 : (31 - __clz((int)(ab & 0x7FFFFFu))) - 149;  // floor(log2)
                const int e = min(max(fl - kEmax, -127), 127);
                sbyte = (uint32_t)(e + 127);
                const float mult = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, a normal float
                const uint32_t xw[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                                         v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
                uint32_t w[8];  // code word q: elements 4q .. 4q+3, element 4q in the low byte
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t a = xw[2 * q], b = xw[2 * q + 1];
                    w[q] = cvt_mx_x2<ELEM>(__fmul_rn(bf16lo(a), mult), __fmul_rn(bf16hi(a), mult)) |
                           (cvt_mx_x2<ELEM>(__fmul_rn(bf16lo(b), mult), __fmul_rn(bf16hi(b), mult)) << 16);
                    if constexpr (WIDEN) w[q] = widen4<ELEM>(w[q]);
                }
                out[0] = make_uint4(w[0], w[1], w[2], w[3]);
                out[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
            uint4* pc = reinterpret_cast<uint4*>(codes + r * k + j * 32);
            pc[0] = out[0];
            pc[1] = out[1];
        }
        scales[sf_offset(r, j, ksf)] = (uint8_t)sbyte;
    }
}

// in may equal out: each thread reads, then writes, its own 16 bytes
__global__ void __launch_bounds__(kMx8Threads) mx6_widen_kernel(int elem, const uint4* in, uint4* out, int64_t n16) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * kMx8Threads + threadIdx.x; i < n16; i += (int64_t)gridDim.x * kMx8Threads) {
        const uint4 v = in[i];
        out[i] = elem == MX_ELEM_E2M3
                     ? make_uint4(widen4<MX_ELEM_E2M3>(v.x), widen4<MX_ELEM_E2M3>(v.y), widen4<MX_ELEM_E2M3>(v.z),
                                  widen4<MX_ELEM_E2M3>(v.w))
                     : make_uint4(widen4<MX_ELEM_E3M2>(v.x), widen4<MX_ELEM_E3M2>(v.y), widen4<MX_ELEM_E3M2>(v.z),
                                  widen4<MX_ELEM_E3M2>(v.w));
    }
}

cudaError_t launch_mx6_widen(int elem, const uint8_t* in, uint8_t* out, int64_t bytes, int sm_count, cudaStream_t s) {
    const int64_t n16 = bytes / 16;
    const int64_t want = (n16 + kMx8Threads - 1) / kMx8Threads;
    const unsigned grid = (unsigned)(want < (int64_t)sm_count * 8 ? (want > 0 ? want : 1) : (int64_t)sm_count * 8);
    mx6_widen_kernel<<<grid, kMx8Threads, 0, s>>>(elem, reinterpret_cast<const uint4*>(in), reinterpret_cast<uint4*>(out),
                                                   n16);
    return cudaGetLastError();
}

cudaError_t launch_mx8_quant(int elem, const uint16_t* x, int64_t rows, int64_t k, uint8_t* codes, uint8_t* scales,
                             int sm_count, cudaStream_t s, bool widen) {
    const int64_t rows_pad = round_up(rows, 128);
    const int64_t ksf = sf_cols_padded(k, 32);
    const int64_t total = rows_pad * ksf;
    const int64_t want = (total + kMx8Threads - 1) / kMx8Threads;
    const unsigned grid = (unsigned)(want < (int64_t)sm_count * 8 ? want : (int64_t)sm_count * 8);
    switch (elem) {
        case MX_ELEM_E4M3:
            mx8_quant_kernel<MX_ELEM_E4M3, false><<<grid, kMx8Threads, 0, s>>>(x, rows, k, rows_pad, ksf, codes, scales);
            break;
        case MX_ELEM_E5M2:
            mx8_quant_kernel<MX_ELEM_E5M2, false><<<grid, kMx8Threads, 0, s>>>(x, rows, k, rows_pad, ksf, codes, scales);
            break;
        case MX_ELEM_E2M3:
            if (widen)
                mx8_quant_kernel<MX_ELEM_E2M3, true><<<grid, kMx8Threads, 0, s>>>(x, rows, k, rows_pad, ksf, codes, scales);
            else
                mx8_quant_kernel<MX_ELEM_E2M3, false><<<grid, kMx8Threads, 0, s>>>(x, rows, k, rows_pad, ksf, codes, scales);
            break;
        case MX_ELEM_E3M2:
            if (widen)
                mx8_quant_kernel<MX_ELEM_E3M2, true><<<grid, kMx8Threads, 0, s>>>(x, rows, k, rows_pad, ksf, codes, scales);
            else
                mx8_quant_kernel<MX_ELEM_E3M2, false><<<grid, kMx8Threads, 0, s>>>(x, rows, k, rows_pad, ksf, codes, scales);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace fp4
