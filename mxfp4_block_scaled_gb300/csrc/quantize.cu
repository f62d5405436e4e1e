// quantize.cu -- bf16 -> NVFP4 / MXFP4 quantisers.
//
// NVFP4 ("vLLM on DGX Spark: technical report", section 6.1 "NVFP4 format"):
// per 16-element K block, s_b = E4M3_rne_satfinite(amax_b / fl(6 s_g)),
// d = fl(s_b * s_g), element = E2M1_rne_satfinite(fl(x / d)), 0 when d == 0.
// MXFP4 (same page, section 6.4): per 32-element block, E8M0 exponent
// e = floor(log2 amax_b) - 2 (clamped to [-127, 127]); element =
// E2M1_rne_satfinite(x * 2^-e) (exact), all-zero blocks give byte 0 and zeros.
//
// Layout of the work: one warp quantises a 256-element K tile of one row; lane
// l holds elements 8l..8l+7 (one 16-byte load), so an NVFP4 block is a lane
// pair and an MXFP4 block four lanes.  Codes leave as one 32-bit store per
// lane (128 contiguous bytes per warp); scales are gathered by shuffles into
// 32-bit words of the MMA layout.  All float operations are single IEEE
// operations (__fdiv_rn / __fmul_rn), matching the CPU oracle bit for bit.
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

namespace fp4 {

constexpr int QT = 256;  // threads per block

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Max over the block of a non-negative value held as uint bits.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
    v = warp_max_u32(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    if (w == 0) {
        v = l < (int)(blockDim.x >> 5) ? red[l] : 0u;
        v = warp_max_u32(v);
        if (l == 0) red[0] = v;
    }
    __syncthreads();
    v = red[0];
    __syncthreads();
    return v;
}

// |bf16| pair maxima: the sign-cleared bit patterns of non-NaN bf16 values
// order like their magnitudes, so a 16-bit unsigned max is an exact abs-max.
__device__ __forceinline__ uint32_t absmax8(const uint4& v, uint32_t m) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
    return m;
}

__global__ void __launch_bounds__(QT) amax_partial_kernel(const uint4* __restrict__ x, int64_t n_vec,
                                                          float* __restrict__ partials) {
    __shared__ uint32_t red[QT / 32];
    pdl_wait();
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * QT;
    int64_t i = (int64_t)blockIdx.x * QT + threadIdx.x;
    for (; i + stride < n_vec; i += 2 * stride) {
        const uint4 a = __ldg(x + i);
        const uint4 b = __ldg(x + i + stride);
        m = absmax8(a, m);
        m = absmax8(b, m);
    }
    if (i < n_vec) m = absmax8(__ldg(x + i), m);
    m = max(m & 0xFFFFu, m >> 16);
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = __uint_as_float(m << 16);
    pdl_launch_dependents();
}

int amax_partials_count(int64_t n_elems) {
    const DeviceInfo* d = current_device();
    const int sms = d ? d->sm_count : 148;
    int64_t want = (n_elems / 8 + QT * 8 - 1) / (QT * 8);  // >= 8 vectors per thread
    if (want < 1) want = 1;
    const int64_t cap = (int64_t)sms * 4;
    return (int)(want < cap ? want : cap);
}

static cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t s,
                             void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_amax_partials(const uint16_t* x, int64_t n_elems, float* partials, int n_part, bool pdl,
                                 cudaStream_t s) {
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    int64_t n_vec = n_elems / 8;
    void* args[] = {(void*)&xv, (void*)&n_vec, (void*)&partials};
    return launch_ex((const void*)amax_partial_kernel, dim3(n_part), dim3(QT), 0, pdl, s, args);
}

// ------------------------------------------------------------- quantiser

template <bool MX>
__global__ void __launch_bounds__(QT) quant_kernel(const QuantLaunch q) {
    __shared__ uint32_t red[QT / 32];
    __shared__ float sh_sg;
    pdl_wait();

    // Per-tensor global scale (modes that have one).
    float sg_tensor = q.static_scale;
    if (!MX && q.sg_mode == SG_PARTIALS) {
        uint32_t m = 0;
        for (int i = threadIdx.x; i < q.n_partials; i += QT) m = max(m, __float_as_uint(q.partials[i]));
        m = block_max_u32(m, red);
        if (threadIdx.x == 0) sh_sg = __fdiv_rn(__uint_as_float(m), 2688.0f);
        __syncthreads();
        sg_tensor = sh_sg;
    }
    if (blockIdx.x == 0) {
        if (q.global_out && threadIdx.x == 0) *q.global_out = MX ? 1.0f : sg_tensor;
        if (!MX && q.sg_mode == SG_EXPERT_AMAX && q.expert_sg_out)
            for (int e = threadIdx.x; e < q.n_experts; e += QT)
                q.expert_sg_out[e] = __fdiv_rn(q.table[e], 2688.0f);
    }

    const int lane = threadIdx.x & 31;
    const int64_t chunks = (q.k + 255) / 256;
    const int64_t ksf_pad = sf_cols_padded(q.k, MX ? 32 : 16);
    const int64_t row_limit = q.rows_dev ? (int64_t)(*q.rows_dev) : q.rows_pad;
    const int64_t total = q.rows_pad * chunks;
    const int64_t warps = (int64_t)gridDim.x * (QT / 32);
    const int64_t kb = q.k / 2;

    for (int64_t item = (int64_t)blockIdx.x * (QT / 32) + (threadIdx.x >> 5); item < total; item += warps) {
        const int64_t r = item / chunks;
        const int64_t c = item - r * chunks;
        if (r >= row_limit) continue;  // warp-uniform
        const int64_t col = c * 256 + lane * 8;
        int64_t src = -1;
        if (r < q.rows) {
            src = r;
            if (q.row_map) {
                const int64_t m = q.row_map[r];
                src = q.row_map_is_mask ? (m >= 0 ? r : -1) : m;
            }
        }
        const bool in = (src >= 0) && (col < q.k);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (in) v = __ldg(reinterpret_cast<const uint4*>(q.x + src * q.x_ld + col));
        const float f[8] = {bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y),
                            bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w)};
        uint32_t am = absmax8(v, 0u);
        am = max(am & 0xFFFFu, am >> 16);
        uint32_t sbyte;
        uint32_t packed = 0;
        if (!MX) {
            am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
            const float amax_b = __uint_as_float(am << 16);
            float sg = sg_tensor;
            if (q.sg_mode == SG_EXPERT_TABLE) sg = q.table[q.tile_expert[r >> 7]];
            else if (q.sg_mode == SG_EXPERT_AMAX) sg = __fdiv_rn(q.table[q.tile_expert[r >> 7]], 2688.0f);
            const float p = __fmul_rn(sg, 6.0f);
            sbyte = 0;
            if (p > 0.0f) sbyte = cvt_e4m3(__fdiv_rn(amax_b, p));
            const float d = __fmul_rn(e4m3_to_f32(sbyte), sg);
            if (d != 0.0f) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    packed |= cvt_e2m1x2(__fdiv_rn(f[2 * i], d), __fdiv_rn(f[2 * i + 1], d)) << (8 * i);
            }
        } else {
            am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
            am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
            const float amax_b = __uint_as_float(am << 16);
            sbyte = 0;
            if (amax_b > 0.0f) {
                const uint32_t u = __float_as_uint(amax_b);
                const int fl = (u >> 23) ? (int)(u >> 23) - 127 : (31 - __clz((int)u)) - 149;
                int e = fl - 2;
                e = e < -127 ? -127 : (e > 127 ? 127 : e);
                sbyte = (uint32_t)(e + 127);
                const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, a normal float here
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    packed |= cvt_e2m1x2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv)) << (8 * i);
            }
        }
        if (in) *reinterpret_cast<uint32_t*>(q.codes + r * kb + col / 2) = packed;
        // Gather four consecutive scale bytes into one word of the MMA layout.
        if (!MX) {
            const int base = lane & ~7;
            const uint32_t s0 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 0);
            const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 2);
            const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 4);
            const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 6);
            if ((lane & 7) == 0)
                *reinterpret_cast<uint32_t*>(q.scales + sf_offset(r, c * 16 + (lane >> 3) * 4, ksf_pad)) =
                    s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
        } else {
            const int base = lane & ~15;
            const uint32_t s0 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 0);
            const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 4);
            const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 8);
            const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, sbyte, base + 12);
            if ((lane & 15) == 0)
                *reinterpret_cast<uint32_t*>(q.scales + sf_offset(r, c * 8 + (lane >> 4) * 4, ksf_pad)) =
                    s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
    }
    pdl_launch_dependents();
}

cudaError_t launch_quant(const QuantLaunch& q, cudaStream_t s) {
    const DeviceInfo* d = current_device();
    const int sms = d ? d->sm_count : 148;
    const int64_t chunks = (q.k + 255) / 256;
    const int64_t total = q.rows_pad * chunks;
    int64_t blocks = (total + (QT / 32) - 1) / (QT / 32);
    const int64_t cap = (int64_t)sms * (2048 / QT);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    QuantLaunch qq = q;
    void* args[] = {(void*)&qq};
    const void* fn = q.fmt == FP4_MXFP4 ? (const void*)quant_kernel<true> : (const void*)quant_kernel<false>;
    return launch_ex(fn, dim3((unsigned)blocks), dim3(QT), 0, q.pdl, s, args);
}

}  // namespace fp4
