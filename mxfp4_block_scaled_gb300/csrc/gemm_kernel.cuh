// gemm_kernel.cuh -- persistent block-scaled FP4 GEMM on tcgen05 (sm_103a).
//
// D[p][q] = sum_k deq(P)[p][k] * deq(Q)[q][k] for two K-major FP4 operands
// with per-16 (NVFP4, UE4M3) or per-32 (MXFP4, UE8M0) block scales, the GEMM
// of "vLLM on DGX Spark: technical report", section 6.1 (value = element x
// block scale x global scale; the global scales leave as one alpha factor).
//
// One CTA per SM, 6 warps:
//   warp 0      TMA producer: per 256-element K block, a 128-row P tile and a
//               BN-row Q tile (128-byte swizzle) plus their scale atoms
//               (plain bulk copies; the MMA layout makes them contiguous).
//   warp 1      TMEM allocator and MMA issuer (one thread): copies the scale
//               atoms smem -> TMEM (tcgen05.cp 32x128b.warpx4) and issues four
//               M=128 x N=BN x K=64 block-scaled MMAs per K block.
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator, alpha, bf16
//               (or the fused MoE epilogues), global stores.
// Pipelines: STAGES smem stages (full/empty mbarriers) and 1-2 TMEM
// accumulator stages (acc_full/acc_empty).  Every wait is bounded.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace fp4 {

template <int BN, bool MX>
struct GemmCfg {
    static constexpr int BM = 128;
    static constexpr int KB_BYTES = 128;            // one K block = 256 fp4 = 128 bytes per row
    static constexpr int SF_CHUNKS = MX ? 2 : 4;    // 512-byte scale atoms per 128 rows per K block
    static constexpr int QCH = BN > 128 ? BN / 128 : 1;
    static constexpr int P_BYTES = BM * KB_BYTES;
    static constexpr int Q_BYTES = BN * KB_BYTES;
    static constexpr int SFP_BYTES = SF_CHUNKS * 512;
    static constexpr int SFQ_BYTES = SF_CHUNKS * 512 * QCH;
    static constexpr int STAGE_BYTES = P_BYTES + Q_BYTES + SFP_BYTES + SFQ_BYTES;
    static constexpr int ACC = BN <= 128 ? 2 : 1;
    static constexpr int SFP_COLS = SF_CHUNKS * 4;
    static constexpr int SFQ_COLS = SF_CHUNKS * 4 * QCH;
    static constexpr int SF_COLS = SFP_COLS + SFQ_COLS;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int ST_SMEM = (SMEM_LIMIT - 1024 - BAR_BYTES) / STAGE_BYTES;
    static constexpr int ST_TMEM = (512 - ACC * BN) / SF_COLS;
    static constexpr int ST_MIN = ST_SMEM < ST_TMEM ? ST_SMEM : ST_TMEM;
    static constexpr int STAGES = ST_MIN < 8 ? ST_MIN : 8;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(STAGES >= 2, "pipeline too shallow");
    static_assert(2 * STAGES + 5 <= BAR_BYTES / 8 - 2, "barrier area too small");
    static_assert(ACC * BN + STAGES * SF_COLS <= 512, "TMEM budget");
};

// Work unit -> tile coordinates.
struct Unit {
    int64_t pt, qt;   // P tile, Q tile (within the expert when grouped)
    int s;            // split index
    int e;            // expert (grouped) or 0
    int64_t p_row0;   // first P row
    int64_t q_row0;   // first Q row in the Q tensor
    int64_t kb0, kb1; // K-block range
};

struct Sched {
    int64_t n_ptiles, n_qtiles, units, kbt, kb_per;
    int splits;
};

template <int BN>
__device__ __forceinline__ Sched make_sched(const GemmLaunch& g) {
    Sched s;
    s.kbt = (g.k + 255) / 256;
    s.splits = g.splits;
    s.kb_per = (s.kbt + g.splits - 1) / g.splits;
    s.n_ptiles = g.grouped ? (int64_t)(*g.n_ptiles_dev) : (g.p_rows_valid + 127) / 128;
    s.n_qtiles = (g.q_rows_valid + BN - 1) / BN;
    s.units = s.n_ptiles * s.n_qtiles * g.splits;
    return s;
}

template <int BN>
__device__ __forceinline__ Unit decode_unit(const GemmLaunch& g, const Sched& sc, int64_t u) {
    Unit w;
    w.s = (int)(u % sc.splits);
    const int64_t r = u / sc.splits;
    w.pt = r % sc.n_ptiles;
    w.qt = r / sc.n_ptiles;
    w.e = g.grouped ? g.tile_expert[w.pt] : 0;
    w.p_row0 = w.pt * 128;
    w.q_row0 = (g.grouped ? (int64_t)w.e * g.q_rows_valid : 0) + w.qt * BN;
    w.kb0 = (int64_t)w.s * sc.kb_per;
    w.kb1 = w.kb0 + sc.kb_per < sc.kbt ? w.kb0 + sc.kb_per : sc.kbt;
    return w;
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

template <int BN, bool MX, int EPI>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                const GemmLaunch g, const WaitCfg wc) {
    using C = GemmCfg<BN, MX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sP = smem;
    uint8_t* sQ = sP + C::STAGES * C::P_BYTES;
    uint8_t* sSFP = sQ + C::STAGES * C::Q_BYTES;
    uint8_t* sSFQ = sSFP + C::STAGES * C::SFP_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sSFQ + C::STAGES * C::SFQ_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* accf = bars + 2 * C::STAGES;
    uint64_t* acce = accf + 2;
    uint64_t* drain = acce + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf + a, 1);
            mbar_init(acce + a, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmP);
        prefetch_tensormap(&tmQ);
    }
    if (warp == 1) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    pdl_wait();
    const Sched sc = make_sched<BN>(g);
    const int64_t ksfc = sc.kbt * C::SF_CHUNKS;                 // scale atoms per 128-row tile
    const int64_t q_chunks_total = (g.q_rows + 127) / 128;      // 128-row scale tiles of Q

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t ph = 0;
            uint32_t issued_ph[C::STAGES];
            bool issued[C::STAGES];
            for (int s = 0; s < C::STAGES; ++s) issued[s] = false, issued_ph[s] = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; u < sc.units && ok; u += gridDim.x) {
                const Unit w = decode_unit<BN>(g, sc, u);
                const uint8_t* sfp = g.p_scales + (w.p_row0 >> 7) * ksfc * 512;
                const int64_t qc0 = w.q_row0 >> 7;
                for (int64_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint32_t bytes = C::P_BYTES + C::Q_BYTES + C::SFP_BYTES;
                    for (int c = 0; c < C::QCH; ++c)
                        if (qc0 + c < q_chunks_total) bytes += C::SF_CHUNKS * 512;
                    mbar_arrive_expect_tx(full + stage, bytes);
                    tma_load_2d(&tmP, full + stage, sP + stage * C::P_BYTES, (int32_t)(kb * 128), (int32_t)w.p_row0);
                    tma_load_2d(&tmQ, full + stage, sQ + stage * C::Q_BYTES, (int32_t)(kb * 128), (int32_t)w.q_row0);
                    bulk_load(sSFP + stage * C::SFP_BYTES, sfp + kb * C::SF_CHUNKS * 512, C::SFP_BYTES, full + stage);
                    for (int c = 0; c < C::QCH; ++c)
                        if (qc0 + c < q_chunks_total)
                            bulk_load(sSFQ + stage * C::SFQ_BYTES + c * C::SF_CHUNKS * 512,
                                      g.q_scales + ((qc0 + c) * ksfc + kb * C::SF_CHUNKS) * 512, C::SF_CHUNKS * 512,
                                      full + stage);
                    issued[stage] = true;
                    issued_ph[stage] = ph;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let every copy already in flight land before the CTA exits.
                WaitCfg w2 = wc;
                volatile int never = 0;
                for (int s = 0; s < C::STAGES; ++s)
                    if (issued[s]) mbar_wait(full + s, issued_ph[s], w2, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_mxf4(128, BN, MX);
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true, any = false;
            for (int64_t u = blockIdx.x; u < sc.units && ok; u += gridDim.x) {
                const Unit w = decode_unit<BN>(g, sc, u);
                if (!mbar_wait(acce + acc, aph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                const uint32_t q_sub = BN < 128 ? (uint32_t)((w.q_row0 & 127) >> 5) : 0u;
                for (int64_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(full + stage, ph, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfp_t = tmem + (uint32_t)(C::ACC * BN + stage * C::SF_COLS);
                    const uint32_t sfq_t = sfp_t + C::SFP_COLS;
#pragma unroll
                    for (int c = 0; c < C::SF_CHUNKS; ++c)
                        tmem_cp_sf(sfp_t + c * 4, sdesc_sf(smem_u32(sSFP + stage * C::SFP_BYTES + c * 512)));
#pragma unroll
                    for (int rc = 0; rc < C::QCH; ++rc)
#pragma unroll
                        for (int c = 0; c < C::SF_CHUNKS; ++c)
                            tmem_cp_sf(sfq_t + (c * C::QCH + rc) * 4,
                                       sdesc_sf(smem_u32(sSFQ + stage * C::SFQ_BYTES + (rc * C::SF_CHUNKS + c) * 512)));
                    const uint32_t pa = smem_u32(sP + stage * C::P_BYTES);
                    const uint32_t qa = smem_u32(sQ + stage * C::Q_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(pa + kk * 32);
                        const uint64_t bd = sdesc_sw128(qa + kk * 32);
                        uint32_t sfa, sfb, id;
                        if constexpr (!MX) {
                            sfa = sfp_t + kk * 4;
                            sfb = sfq_t + kk * 4 * C::QCH + q_sub;
                            id = idesc;
                        } else {
                            sfa = sfp_t + (kk >> 1) * 4;
                            sfb = sfq_t + (kk >> 1) * 4 * C::QCH + q_sub;
                            id = idesc_with_sf_id(idesc, (uint32_t)(kk & 1) * 2u);
                        }
                        mma_mxf4<MX>(d_tmem, ad, bd, id, sfa, sfb, (kb > w.kb0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    mma_commit(empty + stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf + acc);
                if (C::ACC == 2) {
                    acc ^= 1;
                    if (acc == 0) aph ^= 1u;
                } else {
                    aph ^= 1u;
                }
            }
            if (!ok && any) {
                // Wait for the tensor-core ops already issued before TMEM is freed.
                mma_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, wc, &never);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue
        const int qd = warp & 3;  // the TMEM lane quarter this warp may access
        int acc = 0;
        uint32_t aph = 0;
        for (int64_t u = blockIdx.x; u < sc.units; u += gridDim.x) {
            const Unit w = decode_unit<BN>(g, sc, u);
            if (!mbar_wait(accf + acc, aph, wc, abort_flag)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * BN);
            const int64_t prow = w.p_row0 + qd * 32 + lane;  // the P row this thread owns

            if constexpr (EPI == EPI_BF16 || EPI == EPI_BF16_T || EPI == EPI_PARTIAL_T) {
                float alpha = 1.0f;
                if (!MX) alpha = __fmul_rn(g.p_global[0], g.q_global[0]);
                const int64_t q0 = w.qt * BN;  // output column (EPI_BF16) / token (transposed)
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c0, r);
                    tmem_ld_wait();
                    if (prow < g.p_rows_valid) {
                        if constexpr (EPI == EPI_BF16) {
                            uint16_t* o = reinterpret_cast<uint16_t*>(g.out) + prow * g.ldo + q0 + c0;
                            if (q0 + c0 + 32 <= g.q_rows_valid) {
                                uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
                                for (int v = 0; v < 4; ++v) {
                                    uint4 x;
                                    x.x = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r[8 * v + 0])),
                                                      __fmul_rn(alpha, __uint_as_float(r[8 * v + 1])));
                                    x.y = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r[8 * v + 2])),
                                                      __fmul_rn(alpha, __uint_as_float(r[8 * v + 3])));
                                    x.z = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r[8 * v + 4])),
                                                      __fmul_rn(alpha, __uint_as_float(r[8 * v + 5])));
                                    x.w = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r[8 * v + 6])),
                                                      __fmul_rn(alpha, __uint_as_float(r[8 * v + 7])));
                                    o4[v] = x;
                                }
                            } else {
                                for (int i = 0; i < 32; ++i)
                                    if (q0 + c0 + i < g.q_rows_valid) {
                                        __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[i])));
                                        o[i] = *reinterpret_cast<uint16_t*>(&h);
                                    }
                            }
                        } else if constexpr (EPI == EPI_BF16_T) {
                            uint16_t* o = reinterpret_cast<uint16_t*>(g.out);
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int64_t t = q0 + c0 + i;
                                if (t < g.q_rows_valid) {
                                    __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[i])));
                                    o[t * g.ldo + prow] = *reinterpret_cast<uint16_t*>(&h);
                                }
                            }
                        } else {
                            float* o = reinterpret_cast<float*>(g.out) + (int64_t)w.s * g.q_rows_valid * g.p_rows_valid;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int64_t t = q0 + c0 + i;
                                if (t < g.q_rows_valid) o[t * g.p_rows_valid + prow] = __uint_as_float(r[i]);
                            }
                        }
                    }
                }
            } else if constexpr (EPI == EPI_SWIGLU) {
                // Q rows are W13 rows interleaved in groups of 32 (gate, up, gate, up, ...):
                // columns [c0, c0+32) are gate and [c0+32, c0+64) up for the same 32 features.
                const float alpha = __fmul_rn(g.p_global_per_expert ? g.p_global[w.e] : g.p_global[0], g.q_global[w.e]);
                const bool valid = prow < (int64_t)g.row_valid_end[w.pt];
                uint16_t* hrow = reinterpret_cast<uint16_t*>(g.out) + prow * g.ldo;
                uint32_t amax_bits = 0;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 64) {
                    uint32_t rg[32], ru[32];
                    tmem_ld32(tb + c0, rg);
                    tmem_ld32(tb + c0 + 32, ru);
                    tmem_ld_wait();
                    const int64_t f0 = (w.qt * BN + c0) / 2;
                    uint32_t hv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float g0 = __fmul_rn(alpha, __uint_as_float(rg[2 * i]));
                        const float g1 = __fmul_rn(alpha, __uint_as_float(rg[2 * i + 1]));
                        const float u0 = __fmul_rn(alpha, __uint_as_float(ru[2 * i]));
                        const float u1 = __fmul_rn(alpha, __uint_as_float(ru[2 * i + 1]));
                        hv[i] = pack_bf16x2(__fmul_rn(silu_f32(g0), u0), __fmul_rn(silu_f32(g1), u1));
                        amax_bits = __vmaxu2(amax_bits, hv[i] & 0x7FFF7FFFu);
                    }
                    if (valid) {
                        uint4* o4 = reinterpret_cast<uint4*>(hrow + f0);
#pragma unroll
                        for (int v = 0; v < 4; ++v) o4[v] = make_uint4(hv[4 * v], hv[4 * v + 1], hv[4 * v + 2], hv[4 * v + 3]);
                    }
                }
                uint32_t m = valid ? max(amax_bits & 0xFFFFu, amax_bits >> 16) : 0u;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                if (lane == 0 && m) atomicMax(reinterpret_cast<unsigned int*>(g.amax_out) + w.e, m << 16);
            } else if constexpr (EPI == EPI_COMBINE) {
                const float alpha = __fmul_rn(g.p_global[w.e], g.q_global[w.e]);
                const bool valid = prow < (int64_t)g.row_valid_end[w.pt];
                int slot = 0;
                float wt = 0.0f;
                if (valid) {
                    slot = g.row_src[prow];
                    wt = g.slot_weight[slot];
                }
                float* yrow = reinterpret_cast<float*>(g.out) + (int64_t)(slot / g.top_k) * g.ldo + w.qt * BN;
                const float sc = __fmul_rn(wt, alpha);
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + c0, r);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            red_add_v4(yrow + c0 + 4 * v, __fmul_rn(sc, __uint_as_float(r[4 * v])),
                                       __fmul_rn(sc, __uint_as_float(r[4 * v + 1])),
                                       __fmul_rn(sc, __uint_as_float(r[4 * v + 2])),
                                       __fmul_rn(sc, __uint_as_float(r[4 * v + 3])));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce + acc);
            if (C::ACC == 2) {
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            } else {
                aph ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fp4
