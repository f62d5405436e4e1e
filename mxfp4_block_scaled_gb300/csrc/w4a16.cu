// w4a16.cu -- weight-only FP4 linear for decode (W4A16):
//   out[t][r] = bf16(s_gW * sum_k x[t][k] * E2M1(code[r][k]) * s_b[r][k / B])
// with bf16 activations that are not quantised ("vLLM on DGX Spark: technical
// report", section 5.3 "Marlin for NVFP4": FP4 weights dequantised to 16 bits
// and multiplied with 16-bit activations).  E2M1 times the block scale is
// exact in fp32, so the only roundings are the fp32 accumulation and the bf16
// output.
//
// A batch of at most kW4A16MaxM rows makes this a weight stream bounded by
// HBM, so it runs on the CUDA cores: a warp reads four weight rows side by
// side, eight lanes per row, each lane 16 code bytes (32 elements) per
// 256-element step, so a row's step is one contiguous 128-byte read.  The
// activations are staged once per CTA in shared memory as fp32; the eight
// lanes of different k read distinct 16-byte pieces (groups of 32 padded to
// 36 floats, so the eight pieces fall in distinct banks) and the four rows'
// lanes of the same k share them (a broadcast).  A lane holds one row
// (m <= 2) or two (m >= 3), so each activation load serves every row the lane
// holds.  Codes become fp32 through the hardware E2M1-pair conversion;
// products are summed per scale block with packed fp32 FMAs, each block's sum
// is scaled by its block scale, and the eight lanes of a row are summed with
// shuffles.  Row slots are 32 rows apart, so the four rows of a warp read the
// same 16-byte piece of the scale layout.  The grid is persistent (as many
// CTAs as fit), each warp taking groups of rows in turn.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "w4a16.h"

namespace fp4 {

constexpr int kW4Threads = 256;

struct W4A16Args {
    const uint16_t* x;  // bf16 [m][k]
    int m;
    int64_t n, k;
    const uint8_t* w_codes;   // [n][k/2]
    const uint8_t* w_scales;  // MMA layout
    const float* w_global;    // NVFP4: one device fp32
    uint16_t* out;            // bf16 [m][n]
};

// The eight E2M1 codes of word w (element 2j in the low nibble of byte j)
// as four fp32 pairs, one hardware conversion per byte.
__device__ __forceinline__ void e2m1_word_f32(uint32_t w, float2 (&p)[4]) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int q = 0; q < 4; ++q) p[q] = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
}

// Block scales of one lane's 32 elements: NVFP4 the two E4M3 bytes of `v`
// (one conversion for both), MXFP4 the E8M0 byte 2^(b - 127) (byte 0 = 2^-127).
template <bool MX>
__device__ __forceinline__ float2 lane_scales(uint32_t v) {
    if constexpr (MX) {
        const float s = v == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(v << 23);
        return make_float2(s, s);
    } else {
        uint32_t h2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)v));
        return __half22float2(*reinterpret_cast<const __half2*>(&h2));
    }
}

// Activations in shared memory as fp32, 32-element groups padded to 36.
__device__ __forceinline__ int64_t xpad(int64_t k) { return (k >> 5) * 36 + (k & 31); }

constexpr int kW4KLanes = 8;  // lanes per weight row

// MT: the number of activation rows (1..4).
template <bool MX, int MT>
__global__ void __launch_bounds__(kW4Threads, MT <= 2 ? 3 : 2) w4a16_kernel(const W4A16Args a) {
    constexpr int R = MT <= 2 ? 1 : 2;  // weight rows per lane
    constexpr int B = R == 1 ? 4 : 2;   // 256-element steps per unit (two units' codes in flight)
    constexpr int BLK = MX ? 32 : 16;
    constexpr int WPB = BLK / 8;                     // 32-bit code words per scale block
    constexpr int64_t kScaleStep = 256 / BLK / 4 * 512;  // scale-layout bytes per 256-element step
    extern __shared__ __align__(16) float xs[];      // [MT][k/32][36] fp32
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rs = lane / kW4KLanes, kl = lane % kW4KLanes;
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    const int64_t k = a.k, n = a.n;
    const int64_t kp = (k >> 5) * 36;  // padded row of activations
    const int64_t rb = k >> 1;         // code bytes per row
    const int64_t ksf = sf_cols_padded(k, BLK);
    const float g = MX ? 1.0f : a.w_global[0];
    // steps s in which this lane holds elements: s * 256 + kl * 32 < k
    const int my_steps = (int)((k - kl * 32 + 255) >> 8);
    const int steps = (int)((k + 255) >> 8);
    const int nb = (steps + B - 1) / B;  // units per row group
    constexpr int kTasksPerTile = 32 / R;  // row groups per 128-row tile
    const int64_t tasks = (n + 127) / 128 * kTasksPerTile;
    const int64_t wstride = (int64_t)gridDim.x * (kW4Threads / 32);
    // a warp's work is a sequence of units (row group, B steps); the codes
    // and scales of the next unit are loaded before the current one is used
    auto rows_of = [&](int64_t task, int64_t (&row)[R]) {
        // rows tile * 128 + slot * 32 + (task % 32/R) * R + i
#pragma unroll
        for (int i = 0; i < R; ++i) row[i] = task / kTasksPerTile * 128 + rs * 32 + task % kTasksPerTile * R + i;
    };
    auto load_unit = [&](int64_t task, int bi, uint4 (&v)[R][B], uint32_t (&sv)[R][B]) {
        int64_t row[R];
        rows_of(task, row);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const bool live = task < tasks && row[i] < n;
            const int s0 = bi * B;
            const uint8_t* pc = a.w_codes + (live ? row[i] * rb + (int64_t)s0 * 128 + kl * 16 : 0);
            const uint8_t* ps =
                a.w_scales + (live ? sf_offset(row[i], ((int64_t)s0 * 256 + kl * 32) / BLK, ksf) : 0);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                v[i][b] = make_uint4(0u, 0u, 0u, 0u);
                sv[i][b] = 0u;
                if (live && s0 + b < my_steps) {
                    v[i][b] = __ldg(reinterpret_cast<const uint4*>(pc + b * 128));
                    // the scale bytes of the lane's blocks (two NVFP4 from an even column, one MXFP4)
                    sv[i][b] = MX ? (uint32_t)__ldg(ps + b * kScaleStep)
                                  : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(ps + b * kScaleStep));
                }
            }
        }
    };
    int64_t task = (int64_t)blockIdx.x * (kW4Threads / 32) + warp;
    int bi = 0;
    uint4 v[R][B], nv[R][B];
    uint32_t sv[R][B], nsv[R][B];
    load_unit(task, 0, v, sv);  // in flight while the activations are staged
    {
        // activations [MT][k] bf16 -> fp32 in shared memory, 16-byte pieces,
        // eight loads in flight per thread
        const int kx = (int)(k >> 3);  // pieces per activation row
        const int pieces = MT * kx;
        for (int p0 = 0; p0 < pieces; p0 += 8 * kW4Threads) {
            uint4 xv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int p = p0 + j * kW4Threads + (int)threadIdx.x;
                xv[j] = p < pieces ? __ldg(reinterpret_cast<const uint4*>(a.x) + p) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int p = p0 + j * kW4Threads + (int)threadIdx.x;
                if (p < pieces) {
                    const int t = p / kx;
                    float* d = xs + t * kp + xpad((int64_t)(p - t * kx) * 8);
                    *reinterpret_cast<float4*>(d) =
                        make_float4(bf16lo(xv[j].x), bf16hi(xv[j].x), bf16lo(xv[j].y), bf16hi(xv[j].y));
                    *reinterpret_cast<float4*>(d + 4) =
                        make_float4(bf16lo(xv[j].z), bf16hi(xv[j].z), bf16lo(xv[j].w), bf16hi(xv[j].w));
                }
            }
        }
    }
    __syncthreads();

    float2 tot[R][MT];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int t = 0; t < MT; ++t) tot[i][t] = make_float2(0.0f, 0.0f);
    while (task < tasks) {
        int64_t ntask = task;
        int nbi = bi + 1;
        if (nbi == nb) {
            nbi = 0;
            ntask += wstride;
        }
        load_unit(ntask, nbi, nv, nsv);
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int s = bi * B + b;
            if (s >= my_steps) continue;
            const float* xr = xs + (s * 8 + kl) * 36;  // the lane's 32 activations of this step
            float2 sc[R];
#pragma unroll
            for (int i = 0; i < R; ++i) sc[i] = lane_scales<MX>(sv[i][b]);
#pragma unroll
            for (int h = 0; h < 32 / BLK; ++h) {  // scale blocks among the lane's 32 elements
                // two chains per block where fewer than four (row, token) chains run side by side
                constexpr bool kTwoChains = R * MT < 4;
                float2 acc0[R][MT], acc1[R][MT];
                float2(&accb)[R][MT] = kTwoChains ? acc1 : acc0;
#pragma unroll
                for (int i = 0; i < R; ++i)
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        acc0[i][t] = make_float2(0.0f, 0.0f);
                        acc1[i][t] = make_float2(0.0f, 0.0f);
                    }
#pragma unroll
                for (int w = h * WPB; w < (h + 1) * WPB; ++w) {  // 8 elements per code word
                    float4 xa[MT], xb[MT];
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        xa[t] = *reinterpret_cast<const float4*>(xr + t * kp + 8 * w);
                        xb[t] = *reinterpret_cast<const float4*>(xr + t * kp + 8 * w + 4);
                    }
#pragma unroll
                    for (int i = 0; i < R; ++i) {
                        const uint32_t cw = w == 0 ? v[i][b].x : w == 1 ? v[i][b].y : w == 2 ? v[i][b].z : v[i][b].w;
                        float2 p[4];
                        e2m1_word_f32(cw, p);
#pragma unroll
                        for (int t = 0; t < MT; ++t) {
                            acc0[i][t] = __ffma2_rn(make_float2(xa[t].x, xa[t].y), p[0], acc0[i][t]);
                            accb[i][t] = __ffma2_rn(make_float2(xa[t].z, xa[t].w), p[1], accb[i][t]);
                            acc0[i][t] = __ffma2_rn(make_float2(xb[t].x, xb[t].y), p[2], acc0[i][t]);
                            accb[i][t] = __ffma2_rn(make_float2(xb[t].z, xb[t].w), p[3], accb[i][t]);
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const float sb = h == 0 ? sc[i].x : sc[i].y;
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        tot[i][t] = __ffma2_rn(acc0[i][t], make_float2(sb, sb), tot[i][t]);
                        if (kTwoChains) tot[i][t] = __ffma2_rn(acc1[i][t], make_float2(sb, sb), tot[i][t]);
                    }
                }
            }
        }
        if (bi == nb - 1) {  // the row group is complete: sum a row's eight lanes and store
            int64_t row[R];
            rows_of(task, row);
#pragma unroll
            for (int i = 0; i < R; ++i) {
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    float sum = __fadd_rn(tot[i][t].x, tot[i][t].y);
#pragma unroll
                    for (int o = kW4KLanes / 2; o > 0; o >>= 1)
                        sum = __fadd_rn(sum, __shfl_xor_sync(0xFFFFFFFFu, sum, o));
                    if (kl == 0 && row[i] < n) {
                        const __nv_bfloat16 hb = __float2bfloat16_rn(__fmul_rn(g, sum));
                        a.out[(int64_t)t * n + row[i]] = *reinterpret_cast<const uint16_t*>(&hb);
                    }
                    tot[i][t] = make_float2(0.0f, 0.0f);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                v[i][b] = nv[i][b];
                sv[i][b] = nsv[i][b];
            }
        task = ntask;
        bi = nbi;
    }
}

template <bool MX>
static const void* w4a16_fn(int m) {
    switch (m) {
        case 1: return (const void*)w4a16_kernel<MX, 1>;
        case 2: return (const void*)w4a16_kernel<MX, 2>;
        case 3: return (const void*)w4a16_kernel<MX, 3>;
        default: return (const void*)w4a16_kernel<MX, 4>;
    }
}

cudaError_t launch_w4a16(int fmt, const uint16_t* x, int m, int64_t n, int64_t k, const uint8_t* w_codes,
                         const uint8_t* w_scales, const float* w_global, uint16_t* out, cudaStream_t s) {
    W4A16Args a;
    a.x = x;
    a.m = m;
    a.n = n;
    a.k = k;
    a.w_codes = w_codes;
    a.w_scales = w_scales;
    a.w_global = w_global;
    a.out = out;
    const bool mx = fmt == FP4_MXFP4;
    const void* fn = mx ? w4a16_fn<true>(m) : w4a16_fn<false>(m);
    static uint64_t attr_done[2][kW4A16MaxM] = {};  // devices on which each instantiation is opted in
    if (cudaError_t e = set_smem_attr_once(fn, m * (kW4A16MaxK / 32) * 36 * 4, attr_done[mx][m - 1])) return e;
    const size_t smem = (size_t)m * (size_t)(k / 32) * 36 * 4;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaError_t e = cudaGetDevice(&dev)) return e;
    if (cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) return e;
    if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kW4Threads, smem)) return e;
    const int64_t tasks = (n + 127) / 128 * (m <= 2 ? 32 : 16);
    const int64_t need = (tasks + kW4Threads / 32 - 1) / (kW4Threads / 32);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sms * std::max(per_sm, 1)));
    void* args[] = {(void*)&a};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kW4Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace fp4
