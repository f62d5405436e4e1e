// gemm.cu -- launchers of the block-scaled GEMM (dense linear and decode
// variants), the split-K reduction and the instantiation table.
#include <cudaTypedefs.h>
#include <stdio.h>

#include <mutex>

#include "gemm_pair.cuh"

namespace fp4 {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map over code rows [rows][row_bytes] (packed FP4: k/2 bytes; 8-bit
// containers: k); box = box_bytes (64 or 128) x box_rows with the swizzle of
// the same width (the MMA's K-major operand layout).
static bool make_codes_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_bytes, int box_rows,
                           int box_bytes) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over the bf16 output [rows][cols] with row pitch ldo elements
// (ldo % 8 == 0, 16-byte aligned base); box = box_cols (16, 32 or 64) columns
// x 128 rows with the swizzle of the same width as the epilogue's staging.
static bool make_out_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t ldo, int box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ldo * 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, 128u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_cols == 16   ? CU_TENSOR_MAP_SWIZZLE_32B
                    : box_cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                     : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over an fp32 output [rows][cols] with row pitch ldo elements
// (ldo % 4 == 0, 16-byte aligned base); box = 32 columns (128 bytes) x 32
// rows, 128-byte swizzle (one epilogue warp's staging).
static bool make_f32_out_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t ldo) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ldo * 4)};
    cuuint32_t box[2] = {32u, 32u};
    cuuint32_t es[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int64_t gemm_k_blocks(int64_t k) { return (k + 2 * GEMM_KB_BYTES - 1) / (2 * GEMM_KB_BYTES); }

template <int BN, int FK, int EPI, bool MC = false>
static cudaError_t launch_one(const GemmLaunch& g, cudaStream_t s) {
    using C = GemmCfg<BN, FK, epi_staging_bytes<EPI, FK>()>;
    auto kern = gemm_kernel<BN, FK, EPI, MC>;
    static uint64_t attr_done = 0;  // devices on which this instantiation is opted in
    if (cudaError_t e = set_smem_attr_once((const void*)kern, C::SMEM, attr_done)) return e;
    CUtensorMap tmP, tmQ, tmO;
    const int64_t row_bytes = g.k / fk_elems_per_byte<FK>();
    // a CTA pair loads the Q tile in halves (one multicast each)
    if (!make_codes_map(&tmP, g.p_codes, g.p_rows, row_bytes, 128, GEMM_KB_BYTES) ||
        !make_codes_map(&tmQ, g.q_codes, g.q_rows, row_bytes, MC ? BN / 2 : BN, GEMM_KB_BYTES)) {
        set_error("cuTensorMapEncodeTiled failed (rows %lld/%lld, k %lld)", (long long)g.p_rows, (long long)g.q_rows,
                  (long long)g.k);
        return cudaErrorInvalidValue;
    }
    if (EPI == EPI_BF16) {
        if (!make_out_map(&tmO, g.out, g.p_rows_valid, g.q_rows_valid, g.ldo, epi_box_cols<FK>())) {
            set_error("cuTensorMapEncodeTiled failed for the output (%lld x %lld, ldo %lld)",
                      (long long)g.p_rows_valid, (long long)g.q_rows_valid, (long long)g.ldo);
            return cudaErrorInvalidValue;
        }
    } else if (EPI == EPI_DSLOT) {
        // D [p_rows][q_rows_valid] fp32, the expert-sorted padded token rows
        if (!make_f32_out_map(&tmO, g.out, g.p_rows, g.q_rows_valid, g.ldo)) {
            set_error("cuTensorMapEncodeTiled failed for D (%lld x %lld, ldo %lld)", (long long)g.p_rows,
                      (long long)g.q_rows_valid, (long long)g.ldo);
            return cudaErrorInvalidValue;
        }
    } else {
        tmO = tmP;  // unused by the other epilogues
    }
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    int64_t units;
    if (epi_swapped_grouped<EPI>()) {
        // upper bound: every 128-row token tile of the capacity, every sub-tile
        units = ((g.q_rows + 127) / 128) * (128 / BN) * (g.p_rows_valid / 128);
    } else if (g.grouped) {
        // upper bound: every padded 128-row tile of the capacity
        units = ((g.p_rows + 127) / 128) * ((g.q_rows_valid + BN - 1) / BN) * g.splits;
    } else {
        units = ((g.p_rows_valid + 127) / 128) * ((g.q_rows_valid + BN - 1) / BN) * g.splits;
    }
    int64_t grid = d->sm_count;
    if (g.max_ctas > 0 && g.max_ctas < grid) grid = g.max_ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (MC) {
        // pairs of CTAs (units are pairs of P tiles): as many clusters of two
        // as can be resident at once
        static int max_clusters[64];
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
        cfg.attrs = attr;
        cfg.numAttrs = na;
        if (max_clusters[d->device] == 0) {
            cfg.gridDim = dim3((unsigned)(d->sm_count & ~1));
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg) != cudaSuccess || n < 1) {
                cudaGetLastError();
                n = d->sm_count / 2;
            }
            max_clusters[d->device] = n;
        }
        int64_t clusters = grid / 2 < max_clusters[d->device] ? grid / 2 : max_clusters[d->device];
        const int64_t pair_units = units / 2;
        if (pair_units < clusters) clusters = pair_units;
        grid = 2 * clusters;
    } else if (units < grid) {
        grid = units;
    }
    if (grid < 1) return cudaSuccess;
    WaitCfg wc;
    wc.limit_ns = wait_limit_ns();
    wc.err = d->err_word;
    GemmLaunch gg = g;
    void* args[] = {(void*)&tmP, (void*)&tmQ, (void*)&tmO, (void*)&gg, (void*)&wc};
    cfg.gridDim = dim3((unsigned)grid);
    if (g.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    return cudaLaunchKernelExC(&cfg, (const void*)kern, args);
}

// CTA-pair GEMM (prefill): clusters of two CTAs, 256 x 256 output tiles.
template <bool MX>
static cudaError_t launch_pair(const GemmLaunch& g, cudaStream_t s) {
    using C = PairCfg<MX>;
    auto kern = gemm_pair_kernel<MX>;
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    static int max_clusters[64];  // per device: clusters that can be resident at once
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters[d->device] == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
        (void)e;
        cfg.gridDim = dim3((unsigned)(d->sm_count & ~1));
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg);
        if (e != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = d->sm_count / 2;
        }
        max_clusters[d->device] = n;
    }
    CUtensorMap tmP, tmQ, tmO;
    if (!make_codes_map(&tmP, g.p_codes, g.p_rows, g.k / 2, 128, 128) ||
        !make_codes_map(&tmQ, g.q_codes, g.q_rows, g.k / 2, 128, 128) ||
        !make_out_map(&tmO, g.out, g.p_rows_valid, g.q_rows_valid, g.ldo, PairCfg<MX>::BOXC)) {
        set_error("cuTensorMapEncodeTiled failed (rows %lld/%lld, k %lld)", (long long)g.p_rows, (long long)g.q_rows,
                  (long long)g.k);
        return cudaErrorInvalidValue;
    }
    const int64_t units = ((g.p_rows_valid + 255) / 256) * ((g.q_rows_valid + 255) / 256);
    int64_t clusters = max_clusters[d->device];
    if (units < clusters) clusters = units;
    if (clusters < 1) return cudaSuccess;
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    if (g.pdl) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    WaitCfg wc;
    wc.limit_ns = wait_limit_ns();
    wc.err = d->err_word;
    GemmLaunch gg = g;
    void* args[] = {(void*)&tmP, (void*)&tmQ, (void*)&tmO, (void*)&gg, (void*)&wc};
    return cudaLaunchKernelExC(&cfg, (const void*)kern, args);
}

cudaError_t launch_gemm_pair(const GemmLaunch& g, cudaStream_t s) {
    return g.fmt == FP4_MXFP4 ? launch_pair<true>(g, s) : launch_pair<false>(g, s);
}

int gemm_pair_max_clusters() {
    const DeviceInfo* d = current_device();
    return d ? d->sm_count / 2 : 76;
}

cudaError_t launch_gemm_moe(const GemmLaunch& g, cudaStream_t s);  // moe.cu

cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s) {
    if (g.fmt == FMT_MX8) {
        // 8-bit-container MX operands: the dense bf16 epilogue
        if (g.epi == EPI_BF16 && g.bn == 256) return launch_one<256, FK_MX8, EPI_BF16>(g, s);
        if (g.epi == EPI_BF16 && g.bn == 128) return launch_one<128, FK_MX8, EPI_BF16>(g, s);
        set_error("no MX8 GEMM instantiation for epilogue %d, BN %d", g.epi, g.bn);
        return cudaErrorInvalidValue;
    }
    const bool mx = g.fmt == FP4_MXFP4;
    switch (g.epi) {
        case EPI_BF16:
            if (g.bn == 256 && g.mc && !g.grouped && g.splits == 1 && ((g.p_rows_valid + 127) / 128) % 2 == 0)
                return mx ? launch_one<256, FK_MX4, EPI_BF16, true>(g, s) : launch_one<256, FK_NV4, EPI_BF16, true>(g, s);
            if (g.bn == 256)
                return mx ? launch_one<256, FK_MX4, EPI_BF16>(g, s) : launch_one<256, FK_NV4, EPI_BF16>(g, s);
            if (g.bn == 128)
                return mx ? launch_one<128, FK_MX4, EPI_BF16>(g, s) : launch_one<128, FK_NV4, EPI_BF16>(g, s);
            break;
        case EPI_BF16_T:
            if (g.bn == 32)
                return mx ? launch_one<32, FK_MX4, EPI_BF16_T>(g, s) : launch_one<32, FK_NV4, EPI_BF16_T>(g, s);
            if (g.bn == 64)
                return mx ? launch_one<64, FK_MX4, EPI_BF16_T>(g, s) : launch_one<64, FK_NV4, EPI_BF16_T>(g, s);
            break;
        case EPI_PARTIAL:
            if (g.bn == 256)
                return mx ? launch_one<256, FK_MX4, EPI_PARTIAL>(g, s) : launch_one<256, FK_NV4, EPI_PARTIAL>(g, s);
            if (g.bn == 128)
                return mx ? launch_one<128, FK_MX4, EPI_PARTIAL>(g, s) : launch_one<128, FK_NV4, EPI_PARTIAL>(g, s);
            break;
        case EPI_PARTIAL_T:
            if (g.bn == 32)
                return mx ? launch_one<32, FK_MX4, EPI_PARTIAL_T>(g, s) : launch_one<32, FK_NV4, EPI_PARTIAL_T>(g, s);
            if (g.bn == 64)
                return mx ? launch_one<64, FK_MX4, EPI_PARTIAL_T>(g, s) : launch_one<64, FK_NV4, EPI_PARTIAL_T>(g, s);
            break;
        case EPI_SWIGLU:
        case EPI_SWIGLU_T:
        case EPI_DSLOT:
        case EPI_DSLOT_T:
            return launch_gemm_moe(g, s);
    }
    set_error("no GEMM instantiation for epilogue %d, BN %d", g.epi, g.bn);
    return cudaErrorInvalidValue;
}

// Instantiations for the grouped MoE GEMMs live here too (one TU keeps the
// template's code in one place; moe.cu only builds the launch records).
cudaError_t launch_gemm_moe(const GemmLaunch& g, cudaStream_t s) {
    if (g.fmt != FP4_NVFP4) return cudaErrorInvalidValue;
    if (g.epi == EPI_SWIGLU_T && g.bn == 32) return launch_one<32, FK_NV4, EPI_SWIGLU_T>(g, s);
    if (g.epi == EPI_DSLOT_T && g.bn == 32) return launch_one<32, FK_NV4, EPI_DSLOT_T>(g, s);
    if (g.epi == EPI_DSLOT) {
        if (g.bn == 128) return launch_one<128, FK_NV4, EPI_DSLOT>(g, s);
        if (g.bn == 64) return launch_one<64, FK_NV4, EPI_DSLOT>(g, s);
    }
    if (g.epi == EPI_SWIGLU) {
        if (g.bn == 256) return launch_one<256, FK_NV4, EPI_SWIGLU>(g, s);
        if (g.bn == 128) return launch_one<128, FK_NV4, EPI_SWIGLU>(g, s);
        if (g.bn == 64) return launch_one<64, FK_NV4, EPI_SWIGLU>(g, s);
    }
    set_error("no MoE GEMM instantiation for BN %d", g.bn);
    return cudaErrorInvalidValue;
}

// out[t][f] = bf16(alpha * sum_s part[s][t][f]) in split order (deterministic).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4* __restrict__ part, int splits, int64_t mn4,
                                                            const float* ga, const float* gw, int mx,
                                                            uint2* __restrict__ out) {
    pdl_wait();
    pdl_launch_dependents();
    const float alpha = mx ? 1.0f : __fmul_rn(gw[0], ga[0]);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < mn4; i += (int64_t)gridDim.x * blockDim.x) {
        float4 a = part[i];
        for (int s = 1; s < splits; ++s) {
            const float4 b = part[(int64_t)s * mn4 + i];
            a.x = __fadd_rn(a.x, b.x);
            a.y = __fadd_rn(a.y, b.y);
            a.z = __fadd_rn(a.z, b.z);
            a.w = __fadd_rn(a.w, b.w);
        }
        out[i] = make_uint2(pack_bf16x2(__fmul_rn(alpha, a.x), __fmul_rn(alpha, a.y)),
                            pack_bf16x2(__fmul_rn(alpha, a.z), __fmul_rn(alpha, a.w)));
    }
}

cudaError_t launch_splitk_reduce(const float* part, int splits, int64_t m, int64_t n, const float* ga,
                                 const float* gw, bool mx, uint16_t* out, bool pdl, cudaStream_t s) {
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    int64_t mn4 = m * n / 4;
    int64_t blocks = (mn4 + 255) / 256;
    if (blocks > (int64_t)d->sm_count * 8) blocks = (int64_t)d->sm_count * 8;
    if (blocks < 1) blocks = 1;
    const float4* p4 = reinterpret_cast<const float4*>(part);
    uint2* o2 = reinterpret_cast<uint2*>(out);
    int mxi = mx ? 1 : 0;
    void* args[] = {(void*)&p4, (void*)&splits, (void*)&mn4, (void*)&ga, (void*)&gw, (void*)&mxi, (void*)&o2};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, (const void*)splitk_reduce_kernel, args);
}

}  // namespace fp4
