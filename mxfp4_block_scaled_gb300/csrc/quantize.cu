// quantize.cu -- bf16 -> NVFP4 / MXFP4 quantisers.
//
// NVFP4 ("vLLM on DGX Spark: technical report", section 6.1 "NVFP4 format"):
// per 16-element K block, s_b = E4M3_rne_satfinite(amax_b / fl(6 s_g)),
// d = fl(s_b * s_g), element = E2M1_rne_satfinite(fl(x / d)), 0 when d == 0.
// MXFP4 (same page, section 6.4): per 32-element block, E8M0 exponent
// e = floor(log2 amax_b) - 2 (clamped to [-127, 127]); element =
// E2M1_rne_satfinite(x * 2^-e) (exact), all-zero blocks give byte 0 and zeros.
//
// Layout of the work: one thread per scale block (see quant_kernel); the
// per-block arithmetic is in quant_math.cuh.  Every value that decides a code
// or a scale byte is the one single IEEE operations (__fdiv_rn / __fmul_rn)
// give, matching the CPU oracle bit for bit.  Codes come from products with a
// reciprocal where that is proven to give the same code: for every input, when
// the block's divisor passes e2m1_product_exact (one multiply per element), else
// element by element by a bracket, else by correctly rounded divisions.  With
// one global scale per tensor the 128 possible divisors are tabulated per CTA.
#include <stdio.h>

#include "common.cuh"
#include "internal.h"
#include "quant_math.cuh"

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

// Eight 16-byte loads in flight per thread (a thread's loads are one grid
// stride apart, so each load instruction of a warp reads 512 contiguous bytes).
__global__ void __launch_bounds__(QT, 6) amax_partial_kernel(const uint4* __restrict__ x, int64_t n_vec,
                                                             float* __restrict__ partials) {
    __shared__ uint32_t red[QT / 32];
    pdl_wait();
    // the quantiser waits for this grid's completion before reading partials,
    // so it may be scheduled now
    pdl_launch_dependents();
    // Sweep from the end of the tensor to its start, so that the start -- which
    // the quantise pass reads first -- is the most recently cached.
    uint32_t m = 0;
    const int64_t stride = (int64_t)gridDim.x * QT;
    const uint4* xe = x + (n_vec - 1);
    int64_t i = (int64_t)blockIdx.x * QT + threadIdx.x;
    for (; i < n_vec; i += 8 * stride) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            v[u] = i + u * stride < n_vec ? __ldg(xe - (i + u * stride)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < 8; ++u) m = absmax8(v[u], m);
    }
    m = max(m & 0xFFFFu, m >> 16);
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = __uint_as_float(m << 16);
}

int amax_partials_count(int64_t n_elems) {
    const DeviceInfo* d = current_device();
    const int sms = d ? d->sm_count : 148;
    int64_t want = (n_elems / 8 + QT * 8 - 1) / (QT * 8);  // >= 8 vectors per thread
    if (want < 1) want = 1;
    int64_t cap = (int64_t)sms * 6;
    if (cap > 1024) cap = 1024;
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

// One thread per scale block: 16 elements (NVFP4) or 32 (MXFP4) of one row.
// A CTA covers `rpi` rows at a time with `bpt` threads per row (consecutive
// threads take consecutive blocks, so a warp reads a contiguous stretch of the
// row and writes contiguous codes), and walks rows with a grid stride.  Rows
// and blocks past the data (padding of the MMA scale layout) get zero scales.
template <bool MX>
__global__ void __launch_bounds__(QT) quant_kernel(const QuantLaunch q) {
    constexpr int BLK = MX ? 32 : 16;
    constexpr int NV = BLK / 8;  // 16-byte loads per thread
    __shared__ uint32_t red[QT / 32];
    __shared__ float sh_sg;
    __shared__ float2 dtab[128];  // NVFP4, one global scale: divisor entry per scale byte
    pdl_wait();
    // consumers wait for this grid's completion before reading its output, so
    // they may be scheduled now (a GEMM starts streaming its weights)
    pdl_launch_dependents();

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
    const bool dyn_sg = !MX && (q.sg_mode == SG_EXPERT_TABLE || q.sg_mode == SG_EXPERT_AMAX);
    // one global scale: the 128 divisors (a block's byte is below 0x80) and
    // 1/fl(6 s_g) once per CTA
    float p_t = 0.0f, inv_p = 0.0f;
    if (!MX && !dyn_sg) {
        if (threadIdx.x < 128) dtab[threadIdx.x] = nvfp4_divisor(threadIdx.x, sg_tensor, true);
        p_t = __fmul_rn(sg_tensor, 6.0f);
        inv_p = nvfp4_inv_p(p_t);
        __syncthreads();
    }

    const int nb = (int)sf_cols_padded(q.k, BLK);      // scale blocks per row, padding included
    const int kblocks = (int)(q.k / BLK);              // blocks holding data
    const int bpt = nb < QT ? (nb + 31) / 32 * 32 : QT;  // threads per row
    const int rpi = QT / bpt;                           // rows per CTA iteration
    const int ty = threadIdx.x / bpt, tx = threadIdx.x - ty * bpt;
    if (ty >= rpi) return;
    const int64_t row_limit = q.rows_dev ? (int64_t)(*q.rows_dev) : q.rows_pad;
    const int64_t ksf_pad = nb;
    const int64_t rstride = (int64_t)gridDim.x * rpi;

    // Items (row r, block b) of this thread in order; the loads of the next item
    // are issued before the current one is converted (two in flight).
    struct Item {
        int64_t r, src;
        int b;
        uint4 v[NV];
    };
    auto source_row = [&](int64_t r) -> int64_t {
        if (r >= q.rows) return -1;
        if (!q.row_map) return r;
        const int64_t m = q.row_map[r];
        return q.row_map_is_mask ? (m >= 0 ? r : -1) : m;
    };
    auto load = [&](Item& it) {
#pragma unroll
        for (int i = 0; i < NV; ++i) it.v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (it.src >= 0 && it.b < kblocks) {
            const uint4* px = reinterpret_cast<const uint4*>(q.x + it.src * q.x_ld + (int64_t)it.b * BLK);
#pragma unroll
            for (int i = 0; i < NV; ++i) it.v[i] = __ldg(px + i);
        }
    };
    Item cur;
    cur.r = (int64_t)blockIdx.x * rpi + ty;
    cur.b = tx;
    if (cur.r >= row_limit || cur.b >= nb) return;
    cur.src = source_row(cur.r);
    load(cur);
    while (true) {
        Item nxt;
        nxt.r = cur.r;
        nxt.b = cur.b + bpt;
        if (nxt.b >= nb) {
            nxt.b = tx;
            nxt.r += rstride;
        }
        const bool more = nxt.r < row_limit;
        if (more) {
            nxt.src = nxt.r == cur.r ? cur.src : source_row(nxt.r);
            load(nxt);
        }

        // ---- convert the current item
        if (q.skip_masked_rows && cur.src < 0) {
            if (!more) break;
            cur = nxt;
            continue;
        }
        const int64_t r = cur.r;
        const int b = cur.b;
        const bool in = cur.src >= 0 && b < kblocks;
        uint32_t am = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i) am = absmax8(cur.v[i], am);
        const float amax_b = __uint_as_float(max(am & 0xFFFFu, am >> 16) << 16);
        uint32_t sbyte = 0;
        uint32_t w[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) w[i] = 0u;
        if (!MX) {
            float2 e;
            if (!dyn_sg) {
                sbyte = nvfp4_scale_byte(amax_b, p_t, inv_p);
                e = dtab[sbyte];
            } else {
                // the row's expert scale (the row's 128-row tile belongs to one expert)
                const float t = q.table[q.tile_expert[r >> 7]];
                const float sg = q.sg_mode == SG_EXPERT_TABLE ? t : __fdiv_rn(t, 2688.0f);
                const float p = __fmul_rn(sg, 6.0f);
                sbyte = nvfp4_scale_byte(amax_b, p, nvfp4_inv_p(p));
                e = nvfp4_divisor(sbyte, sg, false);
            }
            float f[8];
            unpack8(cur.v[0], f);
            w[0] = nvfp4_word(f, e);
            unpack8(cur.v[1], f);
            w[1] = nvfp4_word(f, e);
        } else if (amax_b > 0.0f) {
            const uint32_t u = __float_as_uint(amax_b);
            const int fl = (u >> 23) ? (int)(u >> 23) - 127 : (31 - __clz((int)u)) - 149;
            int e = fl - 2;
            e = e < -127 ? -127 : (e > 127 ? 127 : e);
            sbyte = (uint32_t)(e + 127);
            const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, a normal float here
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                float f[8];
                unpack8(cur.v[i], f);
                w[i] = cvt_e2m1x8(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                                  __fmul_rn(f[3], inv), __fmul_rn(f[4], inv), __fmul_rn(f[5], inv),
                                  __fmul_rn(f[6], inv), __fmul_rn(f[7], inv));
            }
        }
        if (in) {
            uint8_t* c = q.codes + r * (q.k / 2) + (int64_t)b * (BLK / 2);
            if (MX)
                *reinterpret_cast<uint4*>(c) = make_uint4(w[0], w[1], w[NV > 2 ? 2 : 0], w[NV > 3 ? 3 : 0]);
            else
                *reinterpret_cast<uint2*>(c) = make_uint2(w[0], w[1]);
        }
        q.scales[sf_offset(r, b, ksf_pad)] = (uint8_t)sbyte;

        if (!more) break;
        cur = nxt;
    }
}

// ------------------------------ NVFP4, per-expert scale, real rows of tiles

// The MoE requantisation when padding rows may stay untouched: a CTA takes
// 128-row tiles (one expert each) and only their real rows, so the work
// follows the tokens rather than the padded capacity; the expert's scale is
// read once per tile.  Same arithmetic as quant_kernel's expert modes.
__global__ void __launch_bounds__(QT) quant_tiles_kernel(const QuantLaunch q) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && q.sg_mode == SG_EXPERT_AMAX && q.expert_sg_out)
        for (int e = threadIdx.x; e < q.n_experts; e += QT) q.expert_sg_out[e] = __fdiv_rn(q.table[e], 2688.0f);
    const int nb = (int)sf_cols_padded(q.k, 16);
    const int kblocks = (int)(q.k / 16);
    const int bpt = nb < QT ? (nb + 31) / 32 * 32 : QT;
    const int rpi = QT / bpt;
    const int ty = threadIdx.x / bpt, tx = threadIdx.x - ty * bpt;
    if (ty >= rpi) return;
    const int64_t ntiles = *q.n_tiles_dev;
    const int64_t cb = q.k / 2;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const float tv = q.table[q.tile_expert[t]];
        const float sg = q.sg_mode == SG_EXPERT_TABLE ? tv : __fdiv_rn(tv, 2688.0f);
        const float p = __fmul_rn(sg, 6.0f);
        const float inv_p = nvfp4_inv_p(p);
        const int64_t rend = q.tile_rows_end[t];
        for (int b = tx; b < nb; b += bpt) {
            for (int64_t r0 = t * 128 + ty; r0 < rend; r0 += 4 * rpi) {  // four rows' loads in flight
                uint4 v[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[j][0] = v[j][1] = make_uint4(0u, 0u, 0u, 0u);
                    if (r0 + j * rpi < rend && b < kblocks) {
                        const uint4* px =
                            reinterpret_cast<const uint4*>(q.x + (r0 + j * rpi) * q.x_ld + (int64_t)b * 16);
                        v[j][0] = __ldg(px);
                        v[j][1] = __ldg(px + 1);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t r = r0 + j * rpi;
                    if (r >= rend) break;
                    const uint32_t am = absmax8(v[j][1], absmax8(v[j][0], 0u));
                    const uint32_t sbyte =
                        nvfp4_scale_byte(__uint_as_float(max(am & 0xFFFFu, am >> 16) << 16), p, inv_p);
                    const float2 e = nvfp4_divisor(sbyte, sg, false);
                    float f[8];
                    unpack8(v[j][0], f);
                    const uint32_t w0 = nvfp4_word(f, e);
                    unpack8(v[j][1], f);
                    const uint32_t w1 = nvfp4_word(f, e);
                    if (b < kblocks) *reinterpret_cast<uint2*>(q.codes + r * cb + (int64_t)b * 8) = make_uint2(w0, w1);
                    q.scales[sf_offset(r, b, nb)] = (uint8_t)sbyte;
                }
            }
        }
    }
}

// ------------------------------------- NVFP4, one global scale, rows as given

// E2M1 codes of the 8 elements of v times rd, rounded products (a divisor
// whose table entry proves them exact); paired fp32 multiplies.
__device__ __forceinline__ uint32_t e2m1_word_rd(const uint4& v, float rd) {
    const float2 r2 = make_float2(rd, rd);
    const float2 a = __fmul2_rn(make_float2(bf16lo(v.x), bf16hi(v.x)), r2);
    const float2 b = __fmul2_rn(make_float2(bf16lo(v.y), bf16hi(v.y)), r2);
    const float2 c = __fmul2_rn(make_float2(bf16lo(v.z), bf16hi(v.z)), r2);
    const float2 d = __fmul2_rn(make_float2(bf16lo(v.w), bf16hi(v.w)), r2);
    return cvt_e2m1x8(a.x, a.y, b.x, b.y, c.x, c.y, d.x, d.y);
}

// The codes of a block whose divisor is not proven for the product path
// (bracket or division; rare), out of line.
__device__ __noinline__ uint2 nvfp4_block_slow(uint4 v0, uint4 v1, float2 e) {
    float f[8];
    unpack8(v0, f);
    const uint32_t w0 = nvfp4_word(f, e);
    unpack8(v1, f);
    return make_uint2(w0, nvfp4_word(f, e));
}

constexpr int QU = 4;        // row groups per thread per iteration: all their loads go out first
constexpr int QNV_CTAS = 3;  // resident CTAs per SM (register budget of quant_mx_rows_kernel)
// quant_nv_kernel holds the next QU row groups' loads in flight while it
// converts the current ones (twice the registers): two CTAs per SM
constexpr int QNV_PIPE_CTAS = 2;

// The NVFP4 quantiser for a tensor with one global scale (static, or dynamic
// from the abs-max partials) and no row map: the dense linear's activations,
// the MoE hidden states, weight prepack.  Same thread layout as quant_kernel
// (a thread per 16-element block, `rpi` rows x `bpt` blocks per CTA step);
// a CTA walks a contiguous range of row groups, QU at a time, issuing the next
// QU groups' loads before it converts the current ones (the loads' latency
// runs under the conversion: 38.6 -> 36.5 us for 8192 x 4096, same codes), and
// takes the divisor of each scale byte from its table.
__global__ void __launch_bounds__(QT, QNV_PIPE_CTAS) quant_nv_kernel(const QuantLaunch q) {
    __shared__ uint32_t red[QT / 32];
    __shared__ float sh_sg;
    __shared__ float2 dtab[128];
    if (!q.x_before_wait) {
        pdl_wait();
        pdl_launch_dependents();
    }

    const int nb = (int)sf_cols_padded(q.k, 16);  // scale blocks per row, padding included
    const int kblocks = (int)(q.k / 16);
    const int bpt = nb < QT ? (nb + 31) / 32 * 32 : QT;
    const int rpi = QT / bpt;  // 1, 2, 4 or 8: divides rows_pad (a multiple of 128)
    const int ty = threadIdx.x / bpt, tx = threadIdx.x - ty * bpt;
    // this CTA's row groups (rpi rows each): a contiguous range
    const uint32_t groups = (uint32_t)(q.rows_pad / rpi);
    const uint32_t per = (groups + gridDim.x - 1) / gridDim.x;
    const uint32_t g_begin = blockIdx.x * per;
    const uint32_t g_end = min(groups, g_begin + per);
    const bool active = ty < rpi && g_begin < g_end;
    const uint32_t rows = (uint32_t)q.rows;
    const uint32_t xstep = (uint32_t)(rpi * q.x_ld);  // elements between a thread's rows
    const uint32_t cstep = (uint32_t)(rpi * (q.k / 2));
    const uint32_t tile_sf = (uint32_t)nb * 128u;  // scale bytes per 128-row tile

    uint4 v[QU][2];
    auto load = [&](uint32_t g, uint32_t r, const uint16_t* px, bool bdata) {
#pragma unroll
        for (int j = 0; j < QU; ++j) {
            v[j][0] = v[j][1] = make_uint4(0u, 0u, 0u, 0u);
            if (g + j < g_end && r + j * rpi < rows && bdata) {
                const uint4* pv = reinterpret_cast<const uint4*>(px + j * xstep);
                v[j][0] = __ldg(pv);
                v[j][1] = __ldg(pv + 1);
            }
        }
    };
    // the first batch of rows is in flight while the global scale and the
    // divisor table are formed (neither is needed to load)
    // (and, after the abs-max pass, before the wait for its partials: the
    // loads overlap that pass's tail)
    const uint32_t r_first = g_begin * rpi + ty;
    if (active) load(g_begin, r_first, q.x + (size_t)r_first * (size_t)q.x_ld + (size_t)tx * 16, tx < kblocks);
    if (q.x_before_wait) {
        pdl_wait();  // the partials, and the buffers this grid writes
        pdl_launch_dependents();
    }

    float sg = q.static_scale;
    if (q.sg_mode == SG_PARTIALS) {
        uint32_t m = 0;
        for (int i = threadIdx.x; i < q.n_partials; i += QT) m = max(m, __float_as_uint(q.partials[i]));
        m = block_max_u32(m, red);
        if (threadIdx.x == 0) sh_sg = __fdiv_rn(__uint_as_float(m), 2688.0f);
        __syncthreads();
        sg = sh_sg;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && q.global_out) *q.global_out = sg;
    if (threadIdx.x < 128) dtab[threadIdx.x] = nvfp4_divisor(threadIdx.x, sg, true);
    const float p = __fmul_rn(sg, 6.0f);
    const float inv_p = nvfp4_inv_p(p);
    __syncthreads();
    if (!active) return;

    bool first = true;
    uint4 vn[QU][2];  // the next QU row groups, in flight during the conversion
    for (int b = tx; b < nb; b += bpt) {
        const bool bdata = b < kblocks;
        const uint32_t sf_col = (uint32_t)(b >> 2) * 512u + (uint32_t)(b & 3);
        uint32_t r = r_first;
        const uint16_t* px = q.x + (size_t)r * (size_t)q.x_ld + (size_t)b * 16;
        uint8_t* pc = q.codes + (size_t)r * (size_t)(q.k / 2) + (size_t)b * 8;
        if (!first) load(g_begin, r, px, bdata);  // (the first block's rows went out before the table)
        first = false;
        for (uint32_t g = g_begin; g < g_end; g += QU) {
            const bool more = g + QU < g_end;
            if (more) {
#pragma unroll
                for (int j = 0; j < QU; ++j) {
                    vn[j][0] = vn[j][1] = make_uint4(0u, 0u, 0u, 0u);
                    if (g + QU + j < g_end && r + (QU + j) * rpi < rows && bdata) {
                        const uint4* pv = reinterpret_cast<const uint4*>(px + (QU + j) * xstep);
                        vn[j][0] = __ldg(pv);
                        vn[j][1] = __ldg(pv + 1);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < QU; ++j) {
                if (g + j >= g_end) break;
                const uint32_t rj = r + j * rpi;
                const uint32_t am = absmax8(v[j][1], absmax8(v[j][0], 0u));
                const float amax_b = __uint_as_float(max(am & 0xFFFFu, am >> 16) << 16);
                const uint32_t sbyte = nvfp4_scale_byte(amax_b, p, inv_p);
                const float2 e = dtab[sbyte];
                uint2 w = make_uint2(0u, 0u);
                if (e.y > 0.0f)
                    w = make_uint2(e2m1_word_rd(v[j][0], e.y), e2m1_word_rd(v[j][1], e.y));
                else if (e.x != 0.0f)
                    w = nvfp4_block_slow(v[j][0], v[j][1], e);
                if (rj < rows && bdata) *reinterpret_cast<uint2*>(pc + j * cstep) = w;
                q.scales[(rj >> 7) * tile_sf + ((rj & 31u) << 4) + (((rj >> 5) & 3u) << 2) + sf_col] = (uint8_t)sbyte;
            }
            if (more) {
#pragma unroll
                for (int j = 0; j < QU; ++j) {
                    v[j][0] = vn[j][0];
                    v[j][1] = vn[j][1];
                }
            }
            r += QU * rpi;
            px += QU * xstep;
            pc += QU * cstep;
        }
    }
}

// ------------------------- NVFP4, per-expert scale, every row of the tiles

constexpr int QE_ROWS = 64;  // rows per work item (half a 128-row tile: one expert)

// Rows of 128-row expert tiles quantised with the tile's expert scale, every
// row of the tiles written: the MoE requantisation of h when the grouped
// GEMM2 has tokens on the 128-row side (it reads the padding rows' zero scale
// bytes), and the dispatch with static per-expert scales (row_map gives each
// row's token).  A work item is half a tile: the CTA tabulates the 128
// divisors of the tile's expert scale (as quant_nv_kernel does for a tensor)
// when the expert changes, then takes the item's 64 x nb blocks as a flat
// range, QU per thread per step with the next step's QU loads in flight
// during the conversion (2 CTAs/SM for the registers; the requantisation of h
// at 32768 x 768: 29.5 -> 28.1 us, same codes), with the row and block of each
// step advanced by constants (no division per block).  Rows without a source get
// zero scale bytes and no codes; rows past the device row count are not
// touched.
// Codes and scale bytes equal quant_kernel's expert modes: each divisor entry
// is nvfp4_divisor's, with the product path wherever it is proven.
__global__ void __launch_bounds__(QT, 2) quant_expert_rows_kernel(const QuantLaunch q) {
    __shared__ float2 dtab[128];
    __shared__ int64_t s_x[QE_ROWS];   // element offset of the row's source, -1: zero row, -2: past the rows
    __shared__ int64_t s_c[QE_ROWS];   // byte offset of the row's codes
    __shared__ int64_t s_sf[QE_ROWS];  // byte offset of the row's scale bytes (block 0)
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && q.sg_mode == SG_EXPERT_AMAX && q.expert_sg_out)
        for (int e = threadIdx.x; e < q.n_experts; e += QT) q.expert_sg_out[e] = __fdiv_rn(q.table[e], 2688.0f);
    const int nb = (int)sf_cols_padded(q.k, 16);
    const int kblocks = (int)(q.k / 16);
    const int per_item = QE_ROWS * nb;
    const int64_t row_limit = q.rows_dev ? (int64_t)(*q.rows_dev) : q.rows_pad;
    const int64_t items = (row_limit + QE_ROWS - 1) / QE_ROWS;
    const int64_t cb = q.k / 2;
    const int dq = QT / nb, dr = QT - dq * nb;  // a step of QT blocks: dq rows and dr blocks
    const int t_row = threadIdx.x / nb, t_col = threadIdx.x - t_row * nb;
    int cached = -1;
    float p = 0.0f, inv_p = 0.0f;
    uint4 v[QU][2], vn[QU][2];
    int rj[QU], cj[QU], rn[QU], cn[QU];
    // this thread's next QU blocks of the item: row / block indices, then the loads
    auto load = [&](int base, int& row, int& col) {
#pragma unroll
        for (int j = 0; j < QU; ++j) {
            rn[j] = row;
            cn[j] = col;
            vn[j][0] = vn[j][1] = make_uint4(0u, 0u, 0u, 0u);
            const int64_t xo = base + j * QT < per_item ? s_x[row] : -1;
            if (xo >= 0 && col < kblocks) {
                const uint4* px = reinterpret_cast<const uint4*>(q.x + xo + (int64_t)col * 16);
                vn[j][0] = __ldg(px);
                vn[j][1] = __ldg(px + 1);
            }
            row += dq;
            col += dr;
            if (col >= nb) {
                col -= nb;
                ++row;
            }
        }
    };
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t r0 = it * QE_ROWS;
        const int e = q.tile_expert[it / (128 / QE_ROWS)];
        const float tv = q.table[e];
        __syncthreads();  // the previous item is done with the table and the row offsets
        if (threadIdx.x < QE_ROWS) {
            const int64_t r = r0 + threadIdx.x;
            int64_t xo = -2;
            if (r < row_limit) {
                const int64_t m = r < q.rows ? (int64_t)q.row_map[r] : -1;
                xo = m < 0 ? -1 : (q.row_map_is_mask ? r : m) * q.x_ld;
            }
            s_x[threadIdx.x] = xo;
            s_c[threadIdx.x] = r * cb;
            s_sf[threadIdx.x] = (r >> 7) * (int64_t)(nb >> 2) * 512 + ((r & 31) << 4) + (((r >> 5) & 3) << 2);
        }
        __syncthreads();
        int row = t_row, col = t_col;  // of this thread's next block in the item
        load(threadIdx.x, row, col);   // in flight while the divisor table is formed
        if (e != cached) {             // the same expert for every thread
            const float sg = q.sg_mode == SG_EXPERT_TABLE ? tv : __fdiv_rn(tv, 2688.0f);
            if (threadIdx.x < 128) dtab[threadIdx.x] = nvfp4_divisor(threadIdx.x, sg, true);
            p = __fmul_rn(sg, 6.0f);
            inv_p = nvfp4_inv_p(p);
            cached = e;
            __syncthreads();
        }
        for (int base = threadIdx.x; base < per_item; base += QU * QT) {
#pragma unroll
            for (int j = 0; j < QU; ++j) {
                v[j][0] = vn[j][0];
                v[j][1] = vn[j][1];
                rj[j] = rn[j];
                cj[j] = cn[j];
            }
            if (base + QU * QT < per_item) load(base + QU * QT, row, col);  // the next batch in flight
#pragma unroll
            for (int j = 0; j < QU; ++j) {
                if (base + j * QT >= per_item) break;
                const int64_t xo = s_x[rj[j]];
                if (xo == -2) continue;
                const uint32_t am = absmax8(v[j][1], absmax8(v[j][0], 0u));
                const uint32_t sbyte = nvfp4_scale_byte(__uint_as_float(max(am & 0xFFFFu, am >> 16) << 16), p, inv_p);
                const int c = cj[j];
                if (xo >= 0 && c < kblocks) {
                    const float2 d = dtab[sbyte];
                    uint2 w = make_uint2(0u, 0u);
                    if (d.y > 0.0f)
                        w = make_uint2(e2m1_word_rd(v[j][0], d.y), e2m1_word_rd(v[j][1], d.y));
                    else if (d.x != 0.0f)
                        w = nvfp4_block_slow(v[j][0], v[j][1], d);
                    *reinterpret_cast<uint2*>(q.codes + s_c[rj[j]] + (int64_t)c * 8) = w;
                }
                q.scales[s_sf[rj[j]] + (c >> 2) * 512 + (c & 3)] = (uint8_t)sbyte;
            }
        }
    }
}

// ----------------------------------------------- MXFP4, rows as given

constexpr int QU_MX = 2;  // rows in flight per thread (a 32-element block is four 16-byte loads)

// The MXFP4 quantiser without a row map (activations and weight prepack): the
// layout of quant_nv_kernel with a thread per 32-element block; the scale is
// an exact power of two, so there is no global scale and no divisor table.
__global__ void __launch_bounds__(QT, QNV_CTAS) quant_mx_rows_kernel(const QuantLaunch q) {
    pdl_wait();
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x == 0 && q.global_out) *q.global_out = 1.0f;
    const int nb = (int)sf_cols_padded(q.k, 32);
    const int kblocks = (int)(q.k / 32);
    const int bpt = nb < QT ? (nb + 31) / 32 * 32 : QT;
    const int rpi = QT / bpt;
    const int ty = threadIdx.x / bpt, tx = threadIdx.x - ty * bpt;
    const uint32_t groups = (uint32_t)(q.rows_pad / rpi);
    const uint32_t per = (groups + gridDim.x - 1) / gridDim.x;
    const uint32_t g_begin = blockIdx.x * per;
    const uint32_t g_end = min(groups, g_begin + per);
    if (ty >= rpi || g_begin >= g_end) return;
    const uint32_t rows = (uint32_t)q.rows;
    const uint32_t xstep = (uint32_t)(rpi * q.x_ld);
    const uint32_t cstep = (uint32_t)(rpi * (q.k / 2));
    const uint32_t tile_sf = (uint32_t)nb * 128u;
    for (int b = tx; b < nb; b += bpt) {
        const bool bdata = b < kblocks;
        const uint32_t sf_col = (uint32_t)(b >> 2) * 512u + (uint32_t)(b & 3);
        uint32_t r = g_begin * rpi + ty;
        const uint16_t* px = q.x + (size_t)r * (size_t)q.x_ld + (size_t)b * 32;
        uint8_t* pc = q.codes + (size_t)r * (size_t)(q.k / 2) + (size_t)b * 16;
        for (uint32_t g = g_begin; g < g_end; g += QU_MX) {
            uint4 v[QU_MX][4];
#pragma unroll
            for (int j = 0; j < QU_MX; ++j) {
#pragma unroll
                for (int i = 0; i < 4; ++i) v[j][i] = make_uint4(0u, 0u, 0u, 0u);
                if (g + j < g_end && r + j * rpi < rows && bdata) {
                    const uint4* pv = reinterpret_cast<const uint4*>(px + j * xstep);
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[j][i] = __ldg(pv + i);
                }
            }
#pragma unroll
            for (int j = 0; j < QU_MX; ++j) {
                if (g + j >= g_end) break;
                const uint32_t rj = r + j * rpi;
                uint32_t am = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) am = absmax8(v[j][i], am);
                float inv;
                const uint32_t sbyte = mxfp4_scale_byte(__uint_as_float(max(am & 0xFFFFu, am >> 16) << 16), inv);
                if (rj < rows && bdata)
                    *reinterpret_cast<uint4*>(pc + j * cstep) =
                        make_uint4(mxfp4_codes8(v[j][0], inv), mxfp4_codes8(v[j][1], inv), mxfp4_codes8(v[j][2], inv),
                                   mxfp4_codes8(v[j][3], inv));
                q.scales[(rj >> 7) * tile_sf + ((rj & 31u) << 4) + (((rj >> 5) & 3u) << 2) + sf_col] = (uint8_t)sbyte;
            }
            r += QU_MX * rpi;
            px += QU_MX * xstep;
            pc += QU_MX * cstep;
        }
    }
}

cudaError_t launch_quant(const QuantLaunch& q, cudaStream_t s) {
    const DeviceInfo* d = current_device();
    const int sms = d ? d->sm_count : 148;
    const int blk = q.fmt == FP4_MXFP4 ? 32 : 16;
    if (q.fmt == FP4_NVFP4 && q.skip_masked_rows && q.tile_rows_end && q.n_tiles_dev &&
        (q.sg_mode == SG_EXPERT_TABLE || q.sg_mode == SG_EXPERT_AMAX)) {
        int64_t blocks = q.rows_pad / 128;  // upper bound on the tiles
        if (blocks > (int64_t)sms * 4) blocks = (int64_t)sms * 4;
        if (blocks < 1) blocks = 1;
        QuantLaunch qq = q;
        void* args[] = {(void*)&qq};
        return launch_ex((const void*)quant_tiles_kernel, dim3((unsigned)blocks), dim3(QT), 0, q.pdl, s, args);
    }
    if (q.fmt == FP4_NVFP4 && !q.skip_masked_rows && q.row_map && q.tile_expert &&
        (q.sg_mode == SG_EXPERT_TABLE || q.sg_mode == SG_EXPERT_AMAX)) {
        int64_t blocks = q.rows_pad / QE_ROWS;  // upper bound on the items
        if (blocks > (int64_t)sms * 2) blocks = (int64_t)sms * 2;  // one resident wave
        if (blocks < 1) blocks = 1;
        QuantLaunch qq = q;
        void* args[] = {(void*)&qq};
        return launch_ex((const void*)quant_expert_rows_kernel, dim3((unsigned)blocks), dim3(QT), 0, q.pdl, s, args);
    }
    const int64_t nb16 = sf_cols_padded(q.k, 16);
    // quant_nv_kernel keeps rows, row steps and scale offsets in 32 bits
    const bool fits32 = q.rows_pad < (1LL << 31) && q.x_ld * 8 < (1LL << 32) && q.rows_pad * nb16 < (1LL << 32);
    const bool one_scale = q.fmt == FP4_NVFP4 && (q.sg_mode == SG_STATIC || q.sg_mode == SG_PARTIALS) && !q.row_map &&
                           !q.rows_dev && fits32;
    const int64_t nb32 = sf_cols_padded(q.k, 32);
    if (q.fmt == FP4_MXFP4 && !q.row_map && !q.rows_dev && q.rows_pad < (1LL << 31) && q.x_ld * 8 < (1LL << 32) &&
        q.rows_pad * nb32 < (1LL << 32)) {
        const int64_t bpt = nb32 < QT ? (nb32 + 31) / 32 * 32 : QT;
        const int64_t groups = q.rows_pad / (QT / bpt);
        int64_t blocks = (groups + QU_MX - 1) / QU_MX;
        if (blocks > (int64_t)sms * QNV_CTAS) blocks = (int64_t)sms * QNV_CTAS;
        if (blocks < 1) blocks = 1;
        QuantLaunch qq = q;
        void* args[] = {(void*)&qq};
        return launch_ex((const void*)quant_mx_rows_kernel, dim3((unsigned)blocks), dim3(QT), 0, q.pdl, s, args);
    }
    if (one_scale) {
        const int64_t nb = nb16;
        const int64_t bpt = nb < QT ? (nb + 31) / 32 * 32 : QT;
        const int64_t groups = q.rows_pad / (QT / bpt);
        int64_t blocks = (groups + QU - 1) / QU;
        if (blocks > (int64_t)sms * QNV_PIPE_CTAS) blocks = (int64_t)sms * QNV_PIPE_CTAS;
        if (blocks < 1) blocks = 1;
        QuantLaunch qq = q;
        void* args[] = {(void*)&qq};
        return launch_ex((const void*)quant_nv_kernel, dim3((unsigned)blocks), dim3(QT), 0, q.pdl, s, args);
    }
    const int64_t nb = sf_cols_padded(q.k, blk);
    const int64_t bpt = nb < QT ? (nb + 31) / 32 * 32 : QT;
    const int64_t rpi = QT / bpt;
    int64_t blocks = (q.rows_pad + rpi - 1) / rpi;
    const int64_t cap = (int64_t)sms * 4;  // persistent: one wave at this kernel's occupancy
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    QuantLaunch qq = q;
    void* args[] = {(void*)&qq};
    const void* fn = q.fmt == FP4_MXFP4 ? (const void*)quant_kernel<true> : (const void*)quant_kernel<false>;
    return launch_ex(fn, dim3((unsigned)blocks), dim3(QT), 0, q.pdl, s, args);
}

}  // namespace fp4
