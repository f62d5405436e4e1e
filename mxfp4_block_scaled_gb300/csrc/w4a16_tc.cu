// w4a16_tc.cu -- the weight-only FP4 linear (W4A16) on the tensor cores.
//
// out[t][r] = bf16(s_gW * sum_k x[t][k] * E2M1(code[r][k]) * s_b[r][k / B]),
// the computation of w4a16.cu ("vLLM on DGX Spark: technical report",
// section 5.3 "Marlin for NVFP4": FP4 weights dequantised to 16 bits and
// multiplied with 16-bit activations).  E2M1 times an E4M3 (or E8M0) block
// scale has at most six significant bits and lies in bf16's exponent range,
// so the dequantised weight is exact in bf16; the tensor core forms exact
// products of bf16 operands and sums them in fp32, and s_gW is applied to the
// fp32 sum.  The rounding is therefore the fp32 accumulation's (in the tensor
// core's order) and the one bf16 rounding of the output.
//
// One CTA per 128 weight rows, the whole K; MMA kind::f16 with bf16 A and B,
// M = 128 weight rows, N = 16 activation rows (rows >= m are zero: the TMA
// fills them), K = 16 per instruction:
//   warp 16     weight producer: per 256-element K block one stage of the
//               codes (128 rows x 128 B, 128-byte swizzle) and their scale
//               atoms (bulk copy), from the first instruction (no dependency
//               wait); the dequantisers release a stage as soon as they have
//               read it
//   warp 18     activation producer: the four 64-element boxes (16 rows x
//               128 B) per K block, after the dependency wait
//   warps 0-15  dequantisers: a K block's codes and scales are read into
//               registers (a thread per quarter row of each 64-element
//               sub-block: 4 x 16 codes), then each sub-block becomes a
//               128 x 64 bf16 tile in the MMA's K-major 128-byte-swizzled layout
//   warp 17     TMEM allocation and the MMA issuer (four MMAs per sub-block)
//   warps 0-3   then the epilogue: the 128 x 16 fp32 accumulator, s_gW, bf16 out
// Every wait is bounded; on expiry the role sets the device error word and
// an abort flag that stops the others.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "w4a16.h"

namespace fp4 {

template <bool MX>
struct W4TcCfg {
    static constexpr int N = 16;                           // activation rows on the MMA N side
    static constexpr int SF_CHUNKS = MX ? 2 : 4;           // 512-byte scale atoms per 128 rows per K block
    static constexpr int CODE_BYTES = 128 * 128;           // 128 weight rows x 256 FP4
    static constexpr int SF_BYTES = SF_CHUNKS * 512;
    static constexpr int CSTAGE = CODE_BYTES + 2048;       // codes, then the scale atoms (2 KB slot)
    static constexpr int CST = 6;                          // code stages (released by the dequantisers)
    static constexpr int X_BYTES = 4 * N * 128;            // four 64-element boxes of N bf16 rows
    static constexpr int XST = 4;                          // activation stages (released by the MMAs)
    static constexpr int A_BYTES = 128 * 128;              // 128 rows x 64 bf16
    static constexpr int AST = 4;                          // dequantised weight stages (64-element sub-blocks)
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = 1024 + CST * CSTAGE + XST * X_BYTES + AST * A_BYTES + BAR_BYTES;
    static_assert(CSTAGE % 1024 == 0 && X_BYTES % 1024 == 0, "swizzled tiles are 1024-byte aligned");
    static_assert(2 * CST + 2 * XST + 2 * AST + 4 <= BAR_BYTES / 8, "barrier area too small");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

struct W4TcArgs {
    const uint8_t* w_scales;  // MMA layout
    const float* w_global;    // NVFP4: one device fp32; MXFP4: null
    int m;
    int64_t n, k;
    uint16_t* out;            // bf16 [m][n]
};

// Instruction descriptor of kind::f16 with bf16 A and B, K-major, fp32
// accumulate: bits 4-5 D type (F32 = 1), 7-9 / 10-12 A / B type (BF16 = 1),
// 17-22 N/8, 24-28 M/16.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Eight E2M1 codes (element 2j in the low nibble of byte j) times the block
// scale s, as four bf16 pairs (exact: see the file comment).
__device__ __forceinline__ uint4 dequant8_bf16(uint32_t w, float s) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
        __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, s), __fmul_rn(f.y, s));
        o[q] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// A block-scale byte as fp32: E4M3 (NVFP4) or E8M0 2^(b - 127) (MXFP4, byte 0 = 2^-127).
template <bool MX>
__device__ __forceinline__ float scale_f32(uint32_t b) {
    if constexpr (MX) {
        return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
    } else {
        return e4m3_to_f32(b);
    }
}

constexpr int kW4TcDeqWarps = 16;                      // dequantiser warps 0-15
constexpr int kW4TcThreads = (kW4TcDeqWarps + 3) * 32;  // + weight producer, MMA issuer, activation producer

template <bool MX>
__global__ void __launch_bounds__(kW4TcThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const W4TcArgs a, const WaitCfg wc) {
    using C = W4TcCfg<MX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sC = smem;                            // code stages: codes, scale atoms
    uint8_t* sX = sC + C::CST * C::CSTAGE;         // activation stages
    uint8_t* sA = sX + C::XST * C::X_BYTES;        // dequantised weight tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(sA + C::AST * C::A_BYTES);
    uint64_t* cfull = bars;                        // the stage's weight copies landed
    uint64_t* cempty = cfull + C::CST;             // the 8 dequantiser warps are done with it
    uint64_t* xfull = cempty + C::CST;             // the stage's activation boxes landed
    uint64_t* xempty = xfull + C::XST;             // the MMAs reading them are complete
    uint64_t* afull = xempty + C::XST;             // the tile is written (8 dequantiser warps)
    uint64_t* aempty = afull + C::AST;             // the MMAs reading the tile are complete
    uint64_t* accf = aempty + C::AST;
    uint64_t* drain = accf + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t kbt = (a.k + 255) / 256;
    const int64_t tile = blockIdx.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::CST; ++s) {
            mbar_init(cfull + s, 1);
            mbar_init(cempty + s, kW4TcDeqWarps);
        }
        for (int s = 0; s < C::XST; ++s) {
            mbar_init(xfull + s, 1);
            mbar_init(xempty + s, 1);
        }
        for (int s = 0; s < C::AST; ++s) {
            mbar_init(afull + s, kW4TcDeqWarps);
            mbar_init(aempty + s, 1);
        }
        mbar_init(accf, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
    }
    constexpr int kWProd = kW4TcDeqWarps, kMma = kW4TcDeqWarps + 1, kXProd = kW4TcDeqWarps + 2;
    if (warp == kMma) {
        tmem_alloc(tslot, 32);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_launch_dependents();  // dependents wait for this grid's completion

    if (warp == kWProd || warp == kXProd) {
        if (lane == 0) {
            // ------------------------------------------------ producers
            // the weight codes and scale atoms (no dependency wait: they do not
            // come from the preceding kernels), and the activations
            const bool is_w = warp == kWProd;
            const int nst = is_w ? C::CST : C::XST;
            uint64_t* fb = is_w ? cfull : xfull;
            uint64_t* eb = is_w ? cempty : xempty;
            const int64_t ksfc = kbt * C::SF_CHUNKS;  // scale atoms per 128-row tile
            const uint8_t* sf = a.w_scales + tile * ksfc * 512;
            if (!is_w) pdl_wait();
            int stage = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, issued_ph = 0;
            bool ok = true;
            for (int64_t kb = 0; kb < kbt; ++kb) {
                if (!mbar_wait(eb + stage, ph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                if (is_w) {
                    uint8_t* st = sC + stage * C::CSTAGE;
                    mbar_arrive_expect_tx(fb + stage, C::CODE_BYTES + C::SF_BYTES);
                    tma_load_2d(&tmW, fb + stage, st, (int32_t)(kb * 128), (int32_t)(tile * 128));
                    bulk_load(st + C::CODE_BYTES, sf + kb * C::SF_CHUNKS * 512, C::SF_BYTES, fb + stage);
                } else {
                    uint8_t* st = sX + stage * C::X_BYTES;
                    mbar_arrive_expect_tx(fb + stage, C::X_BYTES);
                    for (int j = 0; j < 4; ++j)
                        tma_load_2d(&tmX, fb + stage, st + j * C::N * 128, (int32_t)(kb * 256 + j * 64), 0);
                }
                issued |= 1u << stage;
                issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                if (++stage == nst) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) {
                // copies in flight land within microseconds; each wait stops at 1 ms
                WaitCfg w2 = wc;
                if (w2.limit_ns > 1000000ull) w2.limit_ns = 1000000ull;
                volatile int never = 0;
                for (int s = 0; s < nst; ++s)
                    if ((issued >> s) & 1u) mbar_wait(fb + s, (issued_ph >> s) & 1u, w2, &never);
            }
        }
    } else if (warp == kMma) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_bf16(128, C::N);
            int xs = 0, as = 0;
            uint32_t xph = 0, aph = 0;
            bool ok = true, any = false;
            for (int64_t kb = 0; kb < kbt && ok; ++kb) {
                if (!mbar_wait(xfull + xs, xph, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t xb = smem_u32(sX + xs * C::X_BYTES);
                for (int j = 0; j < 4; ++j) {
                    if (!mbar_wait(afull + as, aph, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ab = smem_u32(sA + as * C::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem, sdesc_sw128(ab + kk * 32), sdesc_sw128(xb + j * C::N * 128 + kk * 32), idesc,
                                 (kb > 0 || j > 0 || kk > 0) ? 1u : 0u);
                    any = true;
                    mma_commit(aempty + as);
                    if (++as == C::AST) {
                        as = 0;
                        aph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(xempty + xs);
                if (++xs == C::XST) {
                    xs = 0;
                    xph ^= 1u;
                }
            }
            if (ok) mma_commit(accf);
            if (!ok && any) {
                // the tensor-core work already issued finishes before TMEM is freed
                mma_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, wc, &never);
            }
        }
    } else {
        // ---------------------------------------------------- dequantisers
        // thread (r, h, e): weight row r of the tile, 16-byte code piece h and
        // its 8-byte half e of each 64-element sub-block (16 codes, one NVFP4
        // block)
        const int dt = threadIdx.x;
        const int r = dt >> 2, h = (dt >> 1) & 1, e = dt & 1;
        const uint32_t sfrow = (uint32_t)((r & 31) * 16 + (r >> 5) * 4);
        int cs = 0, as = 0;
        uint32_t cph = 0, aph = 0;
        bool ok = true;
        for (int64_t kb = 0; kb < kbt && ok; ++kb) {
            if (!mbar_wait(cfull + cs, cph, wc, abort_flag)) {
                ok = false;
                break;
            }
            const uint32_t st = smem_u32(sC + cs * C::CSTAGE);
            const uint8_t* satoms = sC + cs * C::CSTAGE + C::CODE_BYTES;
            // the K block's codes and block scales into registers, then the stage
            // is released before the conversions
            uint2 c[4];
            float sc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t pa = st + (uint32_t)r * 128u + ((uint32_t)((2 * j + h) ^ (r & 7)) << 4) + 8u * e;
                asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(c[j].x), "=r"(c[j].y) : "r"(pa));
                if constexpr (MX) {
                    const int b = 2 * j + h;  // 32-element block of the K block: atom b / 4
                    sc[j] = scale_f32<true>(satoms[(b >> 2) * 512 + sfrow + (b & 3)]);
                } else {
                    sc[j] = scale_f32<false>(satoms[j * 512 + sfrow + 2 * h + e]);  // block 4j + 2h + e
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty + cs);
            if (++cs == C::CST) {
                cs = 0;
                cph ^= 1u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!mbar_wait(aempty + as, aph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t ab = smem_u32(sA + as * C::A_BYTES) + (uint32_t)r * 128u;
                const uint4 o0 = dequant8_bf16(c[j].x, sc[j]);
                const uint4 o1 = dequant8_bf16(c[j].y, sc[j]);
                sts128(ab + ((uint32_t)((4 * h + 2 * e) ^ (r & 7)) << 4), o0.x, o0.y, o0.z, o0.w);
                sts128(ab + ((uint32_t)((4 * h + 2 * e + 1) ^ (r & 7)) << 4), o1.x, o1.y, o1.z, o1.w);
                fence_proxy_async();  // generic-proxy writes -> visible to the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(afull + as);
                if (++as == C::AST) {
                    as = 0;
                    aph ^= 1u;
                }
            }
        }
        if (warp < 4) {
            // ------------------------------------------------ epilogue (TMEM lane quarter = warp)
            pdl_wait();  // the output buffer may still be read by the preceding kernels
            if (mbar_wait(accf, 0, wc, abort_flag)) {
                tc_fence_after();
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16), v);
                tmem_ld_wait();
                const float alpha = MX ? 1.0f : *a.w_global;
                const int64_t row = tile * 128 + warp * 32 + lane;
                if (row < a.n) {
                    for (int t = 0; t < a.m; ++t) {
                        const __nv_bfloat16 o = __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(v[t])));
                        a.out[(int64_t)t * a.n + row] = *reinterpret_cast<const uint16_t*>(&o);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 32);
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 w4tc_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        tried = true;
    }
    return fn;
}

template <bool MX>
static cudaError_t launch_tc(const uint16_t* x, const uint8_t* w_codes, const W4TcArgs& a, cudaStream_t s) {
    using C = W4TcCfg<MX>;
    auto kern = w4a16_tc_kernel<MX>;
    static uint64_t attr_done = 0;  // devices on which this instantiation is opted in
    if (cudaError_t e = set_smem_attr_once((const void*)kern, C::SMEM, attr_done)) return e;
    auto fn = w4tc_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap tw, tx;
    {
        cuuint64_t dims[2] = {(cuuint64_t)(a.k / 2), (cuuint64_t)a.n};
        cuuint64_t strides[1] = {(cuuint64_t)(a.k / 2)};
        cuuint32_t box[2] = {128u, 128u};
        cuuint32_t es[2] = {1u, 1u};
        if (fn(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w_codes), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            set_error("cuTensorMapEncodeTiled failed for the weights (%lld x %lld)", (long long)a.n, (long long)a.k);
            return cudaErrorInvalidValue;
        }
    }
    {
        // activations [m][k] bf16, boxes of 64 elements x 16 rows (rows >= m read as zero)
        cuuint64_t dims[2] = {(cuuint64_t)a.k, (cuuint64_t)a.m};
        cuuint64_t strides[1] = {(cuuint64_t)(a.k * 2)};
        cuuint32_t box[2] = {64u, (cuuint32_t)C::N};
        cuuint32_t es[2] = {1u, 1u};
        if (fn(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            set_error("cuTensorMapEncodeTiled failed for the activations (%d x %lld)", a.m, (long long)a.k);
            return cudaErrorInvalidValue;
        }
    }
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    WaitCfg wc;
    wc.limit_ns = wait_limit_ns();
    wc.err = d->err_word;
    W4TcArgs aa = a;
    void* args[] = {(void*)&tw, (void*)&tx, (void*)&aa, (void*)&wc};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.n + 127) / 128));
    cfg.blockDim = dim3(kW4TcThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, (const void*)kern, args);
}

cudaError_t launch_w4a16_tc(int fmt, const uint16_t* x, int m, int64_t n, int64_t k, const uint8_t* w_codes,
                            const uint8_t* w_scales, const float* w_global, uint16_t* out, cudaStream_t s) {
    W4TcArgs a;
    a.w_scales = w_scales;
    a.w_global = w_global;
    a.m = m;
    a.n = n;
    a.k = k;
    a.out = out;
    return fmt == FP4_MXFP4 ? launch_tc<true>(x, w_codes, a, s) : launch_tc<false>(x, w_codes, a, s);
}

}  // namespace fp4
