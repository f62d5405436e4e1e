// gemm_pair.cuh -- block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same arithmetic as gemm_kernel.cuh (D = deq(P) . deq(Q)^T, alpha and bf16
// in the epilogue), for large problems.  Two CTAs of a cluster compute one
// 256 x 256 output tile with M=256 x N=256 x K=64 MMAs issued by the even CTA:
// each CTA holds 128 rows of the P tile and 128 rows (one half) of the Q tile
// in its shared memory and its 128 output rows in its Tensor Memory, so a
// K block costs each SM 38 KB of shared memory instead of 54 KB, and five
// stages fit.
//
// Per CTA, 16 warps: 0-3 scale writers (the CTA's own P scales and all 256
// rows of Q scales into its own TMEM), 4 and 6 TMA producers (P half, Q half),
// 5 TMEM allocation (collective over the pair) and, in the even CTA, the MMA
// issuer, 8-15 epilogue.  Cross-CTA edges:
//   - a stage may be consumed once both CTAs' scale writers have seen their
//     own data land and stored the scales: they arrive on the even CTA's
//     `sfr` barrier (4 + 4 arrivals);
//   - the MMA commit is multicast to the `empty` and `acc_full` barriers of
//     both CTAs;
//   - both CTAs' epilogues release the accumulator on the even CTA's
//     `acc_empty` barrier (8 + 8 arrivals).
// Every wait is bounded; the CTAs meet at cluster barriers before the first
// remote arrive and before the Tensor Memory is freed.
#pragma once

#include "gemm_kernel.cuh"

namespace fp4 {

template <bool MX>
struct PairCfg {
    static constexpr int BN = 256;                 // pair tile width (N); each CTA holds BN / 2 Q rows
    static constexpr int KB_BYTES = 128;
    static constexpr int SF_CHUNKS = MX ? 2 : 4;
    static constexpr int P_BYTES = 128 * KB_BYTES;
    static constexpr int Q_BYTES = 128 * KB_BYTES;
    static constexpr int SFP_BYTES = SF_CHUNKS * 512;
    static constexpr int SFQ_BYTES = SF_CHUNKS * 512 * 2;  // all 256 Q rows
    static constexpr int STAGE_BYTES = P_BYTES + Q_BYTES + SFP_BYTES + SFQ_BYTES;
    static constexpr int SFP_COLS = SF_CHUNKS * 4;
    static constexpr int SFQ_COLS = SF_CHUNKS * 4 * 2;
    static constexpr int SF_COLS = SFP_COLS + SFQ_COLS;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int BOXC = 64;                                // bf16 epilogue box: 128 x 64
    static constexpr int STG = 2 * epi_buffer_bytes<BOXC>();       // bf16 epilogue staging
    static constexpr int ST_SMEM = (SMEM_LIMIT - 1024 - BAR_BYTES - STG) / STAGE_BYTES;
    static constexpr int ST_TMEM = (512 - BN) / SF_COLS;
    static constexpr int ST_MIN = ST_SMEM < ST_TMEM ? ST_SMEM : ST_TMEM;
    static constexpr int STAGES = ST_MIN < 8 ? ST_MIN : 8;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + STG + BAR_BYTES;
    static_assert(STAGE_BYTES % 1024 == 0, "staging must stay 1024-byte aligned");
    static_assert(3 * STAGES + 5 <= BAR_BYTES / 8 - 2, "barrier area too small");
    static_assert(BN + STAGES * SF_COLS <= 512, "TMEM budget");
};

template <bool MX>
__global__ void __launch_bounds__(512, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmO, const GemmLaunch g, const WaitCfg wc) {
    using C = PairCfg<MX>;
    constexpr int BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sP = smem;
    uint8_t* sQ = sP + C::STAGES * C::P_BYTES;
    uint8_t* sSFP = sQ + C::STAGES * C::Q_BYTES;
    uint8_t* sSFQ = sSFP + C::STAGES * C::SFP_BYTES;
    uint8_t* sStg = sSFQ + C::STAGES * C::SFQ_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + C::STG);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* sfr = bars + 2 * C::STAGES;
    uint64_t* accf = bars + 3 * C::STAGES;
    uint64_t* acce = accf + 1;
    uint64_t* drain = acce + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + s, 2);   // this CTA's two producers
            mbar_init(empty + s, 1);  // the pair's MMA commit
            mbar_init(sfr + s, 8);    // scale writers of both CTAs (used in the even CTA)
        }
        mbar_init(accf, 1);
        mbar_init(acce, 16);          // epilogue warps of both CTAs (used in the even CTA)
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmP);
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmO);
    }
    if (warp == 5) {
        tmem_alloc_pair(tslot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tslot;

    pdl_wait();
    const int64_t kbt = (g.k + 255) / 256;
    const int64_t ksfc = kbt * C::SF_CHUNKS;                 // scale atoms per 128-row tile
    const int64_t n_pm = (g.p_rows_valid + 255) / 256;       // 256-row pair tiles of P
    const int64_t n_qt = (g.q_rows_valid + BN - 1) / BN;
    const int64_t units = n_pm * n_qt;
    const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const int64_t q_chunks_total = (g.q_rows + 127) / 128;
    const int64_t p_rows_pad = (g.p_rows + 127) / 128 * 128;  // rows of the P scale buffer
    const uint32_t sfr_leader = mapa_shared(smem_u32(sfr), 0);
    const uint32_t acce_leader = mapa_shared(smem_u32(acce), 0);

    if (warp < 4) {
        // ---------------------------------------------------- scale writers
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int64_t u = cid; u < units && ok; u += ncl) {
            for (int64_t kb = 0; kb < kbt; ++kb) {
                if (!mbar_wait(full + stage, ph, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sfp_t = tmem + lane_base + (uint32_t)(BN + stage * C::SF_COLS);
                const uint32_t sfq_t = sfp_t + C::SFP_COLS;
                const uint32_t sp = smem_u32(sSFP + stage * C::SFP_BYTES) + lane * 16;
                const uint32_t sq = smem_u32(sSFQ + stage * C::SFQ_BYTES) + lane * 16;
#pragma unroll
                for (int c = 0; c < C::SF_CHUNKS; ++c) tmem_st4(sfp_t + c * 4, lds128(sp + c * 512));
#pragma unroll
                for (int rc = 0; rc < 2; ++rc)
#pragma unroll
                    for (int c = 0; c < C::SF_CHUNKS; ++c)
                        tmem_st4(sfq_t + (c * 2 + rc) * 4, lds128(sq + (rc * C::SF_CHUNKS + c) * 512));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                // this CTA's operands of the stage have landed and its scales are in TMEM
                if (lane == 0) mbar_arrive_cluster(sfr_leader + (uint32_t)(stage * 8));
                if (++stage == C::STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 4 || warp == 6) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producers
            const bool is_p = warp == 4;
            int stage = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, issued_ph = 0;
            bool ok = true;
            for (int64_t u = cid; u < units && ok; u += ncl) {
                const int64_t pm = u % n_pm, qt = u / n_pm;
                const int64_t p_row0 = pm * 256 + 128 * rank;
                const int64_t q_row0 = qt * BN + 128 * rank;  // this CTA's half of the Q tile
                const int64_t qc0 = qt * 2;                     // both 128-row scale chunks of the Q tile
                const uint8_t* sfp = g.p_scales + (p_row0 >> 7) * ksfc * 512;
                for (int64_t kb = 0; kb < kbt; ++kb) {
                    if (!mbar_wait_cluster(empty + stage, ph ^ 1u, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (is_p) {
                        // a half tile wholly past the data has no scale atoms in memory
                        // (its TMA box is zero-filled; its output rows are not stored)
                        const bool p_has = p_row0 < p_rows_pad;
                        mbar_arrive_expect_tx(full + stage, C::P_BYTES + (p_has ? C::SFP_BYTES : 0));
                        tma_load_2d(&tmP, full + stage, sP + stage * C::P_BYTES, (int32_t)(kb * 128), (int32_t)p_row0);
                        if (p_has)
                            bulk_load(sSFP + stage * C::SFP_BYTES, sfp + kb * C::SF_CHUNKS * 512, C::SFP_BYTES,
                                      full + stage);
                    } else {
                        uint32_t bytes = C::Q_BYTES;
                        for (int c = 0; c < 2; ++c)
                            if (qc0 + c < q_chunks_total) bytes += C::SF_CHUNKS * 512;
                        mbar_arrive_expect_tx(full + stage, bytes);
                        tma_load_2d(&tmQ, full + stage, sQ + stage * C::Q_BYTES, (int32_t)(kb * 128), (int32_t)q_row0);
                        for (int c = 0; c < 2; ++c)
                            if (qc0 + c < q_chunks_total)
                                bulk_load(sSFQ + stage * C::SFQ_BYTES + c * C::SF_CHUNKS * 512,
                                          g.q_scales + ((qc0 + c) * ksfc + kb * C::SF_CHUNKS) * 512,
                                          C::SF_CHUNKS * 512, full + stage);
                    }
                    issued |= 1u << stage;
                    issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                WaitCfg w2 = wc;
                volatile int never = 0;
                for (int s = 0; s < C::STAGES; ++s)
                    if ((issued >> s) & 1u) mbar_wait(full + s, (issued_ph >> s) & 1u, w2, &never);
            }
        }
    } else if (warp == 5) {
        if (leader && lane == 0) {
            // ------------------------------------------------ MMA issuer (even CTA)
            const uint32_t idesc = idesc_mxf4(256, BN, MX);
            int stage = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true, any = false;
            for (int64_t u = cid; u < units && ok; u += ncl) {
                if (!mbar_wait_cluster(acce, aph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int64_t kb = 0; kb < kbt; ++kb) {
                    if (!mbar_wait(full + stage, ph, wc, abort_flag) ||
                        !mbar_wait_cluster(sfr + stage, ph, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfp_t = tmem + (uint32_t)(BN + stage * C::SF_COLS);
                    const uint32_t sfq_t = sfp_t + C::SFP_COLS;
                    const uint32_t pa = smem_u32(sP + stage * C::P_BYTES);
                    const uint32_t qa = smem_u32(sQ + stage * C::Q_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(pa + kk * 32);
                        const uint64_t bd = sdesc_sw128(qa + kk * 32);
                        uint32_t sfa, sfb, id;
                        if constexpr (!MX) {
                            sfa = sfp_t + kk * 4;
                            sfb = sfq_t + kk * 8;
                            id = idesc;
                        } else {
                            sfa = sfp_t + (kk >> 1) * 4;
                            sfb = sfq_t + (kk >> 1) * 8;
                            id = idesc_with_sf_id(idesc, (uint32_t)(kk & 1) * 2u);
                        }
                        mma_mxf4_pair<MX>(tmem, ad, bd, id, sfa, sfb, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    mma_commit_pair_mc(empty + stage, (uint16_t)3);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_mc(accf, (uint16_t)3);
                aph ^= 1u;
            }
            if (!ok && any) {
                mma_commit_pair_mc(drain, (uint16_t)1);
                volatile int never = 0;
                mbar_wait(drain, 0, wc, &never);
            }
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------- epilogue
        constexpr int CPW = BN / 2;
        constexpr int NLD = CPW / 32;
        const int qd = warp & 3;
        const int wg = (warp - 8) >> 2;
        const int c_begin = wg * CPW;
        bool store_pending = false;
        uint32_t aph = 0;
        for (int64_t u = cid; u < units; u += ncl) {
            if (!mbar_wait_cluster(accf, aph, wc, abort_flag)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)c_begin;
            const float alpha = MX ? 1.0f : __fmul_rn(g.p_global[0], g.q_global[0]);
            uint32_t pk[NLD][16];
#pragma unroll
            for (int j = 0; j < NLD; ++j) {
                uint32_t r[32];
                tmem_ld32(tb + j * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[j][i] = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r[2 * i])),
                                           __fmul_rn(alpha, __uint_as_float(r[2 * i + 1])));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader);
            aph ^= 1u;
            const int64_t pm = u % n_pm, qt = u / n_pm;
            epi_store_bf16<NLD, C::BOXC>(&tmO, smem_u32(sStg) + (uint32_t)(wg * epi_buffer_bytes<C::BOXC>()), pk, qd, lane,
                                1u + (uint32_t)wg, qt * BN + c_begin, pm * 256 + 128 * rank, g.q_rows_valid,
                                g.p_rows_valid, store_pending);
        }
        if (store_pending) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the pair's MMAs and TMEM reads are done in both CTAs
    pdl_launch_dependents();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace fp4
