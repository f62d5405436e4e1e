// gemm_pair.cuh -- block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same arithmetic as gemm_kernel.cuh (D = deq(P) . deq(Q)^T, alpha and bf16
// in the epilogue), for large problems.  Two CTAs of a cluster compute one
// 256 x 256 output tile with M=256 x N=256 x K=64 MMAs issued by the even CTA:
// each CTA holds 128 rows of the P tile and 128 rows (one half) of the Q tile
// in its shared memory and its 128 output rows in its Tensor Memory.  Per K
// block an SM's shared memory takes 32 KB of operand tiles and serves 32 KB of
// MMA operand reads (the one-CTA kernel: 48 + 48 KB), the traffic that bounds
// the one-CTA kernel on large problems.
//
// Per CTA, 16 warps: 0-3 scale writers (the CTA's own P scales and all 256
// rows of Q scales into its own TMEM), 4 and 6 operand TMA producers (P half,
// Q half), 7 scale-atom producer, 5 TMEM allocation (collective over the pair)
// and, in the even CTA, the MMA issuer, 8-15 epilogue.  The even CTA's `full`
// barrier of a stage completes when
//   - the operand tiles of both CTAs have landed: the odd CTA's TMA loads
//     count their bytes on the even CTA's barrier (cta_group::2 copies), and
//     the even CTA's producers expect the bytes of both, and
//   - the scale writers of both CTAs (4 + 4 arrivals) stored the stage's
//     scales into their TMEM.
// Scale atoms travel on a ring of their own (per CTA), so the writers fill a
// stage's TMEM columns as soon as the previous MMAs on that stage are done,
// ahead of the operand tiles.  The MMA commit is multicast to the `empty` and
// `acc_full` barriers of both CTAs; both CTAs' epilogues release the
// accumulator on the even CTA's `acc_empty` barrier.  Every wait is bounded;
// the CTAs meet at cluster barriers before the first remote arrive or copy and
// before the Tensor Memory is freed.  Waits on barriers completed by the
// multicast MMA commit poll at CTA scope; the MMA issuer's waits on barriers
// with remote arrivals (full, acc_empty) poll with cluster-scope acquire.
#pragma once

#include "gemm_kernel.cuh"

namespace fp4 {

template <bool MX>
struct PairCfg {
    static constexpr int BN = 256;  // pair tile width (N); each CTA holds BN / 2 Q rows
    static constexpr int KB_BYTES = 128;
    static constexpr int SF_CHUNKS = MX ? 2 : 4;
    static constexpr int P_BYTES = 128 * KB_BYTES;
    static constexpr int Q_BYTES = 128 * KB_BYTES;
    static constexpr int OP_BYTES = P_BYTES + Q_BYTES;
    static constexpr int SFP_BYTES = SF_CHUNKS * 512;
    static constexpr int SFQ_BYTES = SF_CHUNKS * 512 * 2;  // all 256 Q rows
    static constexpr int SF_BYTES = SFP_BYTES + SFQ_BYTES;
    static constexpr int SFP_COLS = SF_CHUNKS * 4;
    static constexpr int SFQ_COLS = SF_CHUNKS * 4 * 2;
    static constexpr int SF_COLS = SFP_COLS + SFQ_COLS;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int BOXC = epi_box_cols<MX>();           // bf16 epilogue box: 128 x BOXC
    static constexpr int STG = 2 * epi_buffer_bytes<BOXC>();  // bf16 epilogue staging
    static constexpr int BUDGET = SMEM_LIMIT - 2048 - BAR_BYTES - STG;
    static constexpr int ST_SMEM = (BUDGET - 2 * SF_BYTES) / OP_BYTES;
    static constexpr int ST_TMEM = (512 - BN) / SF_COLS;
    static constexpr int ST_MIN = ST_SMEM < ST_TMEM ? ST_SMEM : ST_TMEM;
    static constexpr int STAGES = ST_MIN < 8 ? ST_MIN : 8;
    static constexpr int SS_FIT = (BUDGET - STAGES * OP_BYTES) / SF_BYTES;
    static constexpr int SSLOTS = SS_FIT < STAGES ? SS_FIT : STAGES;
    static constexpr int STG_OFFSET = (STAGES * OP_BYTES + SSLOTS * SF_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM = 1024 + STG_OFFSET + STG + BAR_BYTES;
    static_assert(STAGES >= 2 && SSLOTS >= 2, "pipeline too shallow");
    static_assert(2 * STAGES + 2 * SSLOTS + 5 <= BAR_BYTES / 8 - 2, "barrier area too small");
    static_assert(BN + STAGES * SF_COLS <= 512, "TMEM budget");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
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
    uint8_t* sSFP = sQ + C::STAGES * C::Q_BYTES;  // scale ring (SSLOTS slots)
    uint8_t* sSFQ = sSFP + C::SSLOTS * C::SFP_BYTES;
    uint8_t* sStg = smem + C::STG_OFFSET;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + C::STG);
    uint64_t* full = bars;                   // used in the even CTA
    uint64_t* empty = bars + C::STAGES;      // both CTAs (multicast MMA commit)
    uint64_t* sfull = bars + 2 * C::STAGES;  // scale atoms of the slot landed (own CTA)
    uint64_t* sempty = sfull + C::SSLOTS;    // the writers are done with the slot (own CTA)
    uint64_t* accf = sempty + C::SSLOTS;     // both CTAs (multicast MMA commit)
    uint64_t* acce = accf + 1;               // used in the even CTA
    uint64_t* drain = acce + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // even CTA: its two producers (expecting both CTAs' bytes) + 4 + 4 scale writers
            mbar_init(full + s, 10);
            mbar_init(empty + s, 1);
        }
        for (int s = 0; s < C::SSLOTS; ++s) {
            mbar_init(sfull + s, 1);
            mbar_init(sempty + s, 4);
        }
        mbar_init(accf, 1);
        mbar_init(acce, 16);  // epilogue warps of both CTAs (used in the even CTA)
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
    cluster_sync();  // the peer's barriers are initialised before any remote arrive or copy
    tc_fence_after();
    const uint32_t tmem = *tslot;

    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion before reading its output
    const int64_t kbt = (g.k + 255) / 256;
    const int64_t ksfc = kbt * C::SF_CHUNKS;            // scale atoms per 128-row tile
    const int64_t n_pm = (g.p_rows_valid + 255) / 256;  // 256-row pair tiles of P
    const int64_t n_qt = (g.q_rows_valid + BN - 1) / BN;
    const int64_t units = n_pm * n_qt;
    const int64_t cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
    const int64_t q_chunks_total = (g.q_rows + 127) / 128;
    const int64_t p_rows_pad = (g.p_rows + 127) / 128 * 128;  // rows of the P scale buffer
    const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
    const uint32_t acce_leader = mapa_shared(smem_u32(acce), 0);

    if (warp < 4) {
        // ---------------------------------------------------- scale writers
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int stage = 0, slot = 0;
        uint32_t ph = 0, sph = 0;
        bool ok = true;
        for (int64_t u = cid; u < units && ok; u += ncl) {
            for (int64_t kb = 0; kb < kbt; ++kb) {
                // the slot's atoms are in smem, and the MMAs of the stage's
                // previous round (which read these TMEM columns) are complete
                if (!mbar_wait(sfull + slot, sph, wc, abort_flag) ||
                    !mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sfp_t = tmem + lane_base + (uint32_t)(BN + stage * C::SF_COLS);
                const uint32_t sfq_t = sfp_t + C::SFP_COLS;
                const uint32_t sp = smem_u32(sSFP + slot * C::SFP_BYTES) + lane * 16;
                const uint32_t sq = smem_u32(sSFQ + slot * C::SFQ_BYTES) + lane * 16;
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
                if (lane == 0) {
                    mbar_arrive_cluster(full_leader + (uint32_t)(stage * 8));
                    mbar_arrive(sempty + slot);
                }
                if (++stage == C::STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
                if (++slot == C::SSLOTS) {
                    slot = 0;
                    sph ^= 1u;
                }
            }
        }
    } else if (warp == 4 || warp == 6 || warp == 7) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producers
            // warp 4: this CTA's P half, warp 6: its Q half (both counted on the
            // even CTA's full barrier), warp 7: the scale atoms (own ring).
            const bool is_p = warp == 4, is_sf = warp == 7;
            const int nst = is_sf ? C::SSLOTS : C::STAGES;
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
                // a P half wholly past the data has no scale atoms in memory (its
                // operand box is zero-filled by the TMA; its rows are not stored)
                const bool p_has = p_row0 < p_rows_pad;
                for (int64_t kb = 0; kb < kbt; ++kb) {
                    if (is_sf) {
                        if (!mbar_wait(sempty + stage, ph ^ 1u, wc, abort_flag)) {
                            ok = false;
                            break;
                        }
                        uint32_t bytes = p_has ? C::SFP_BYTES : 0;
                        for (int c = 0; c < 2; ++c)
                            if (qc0 + c < q_chunks_total) bytes += C::SF_CHUNKS * 512;
                        mbar_arrive_expect_tx(sfull + stage, bytes);
                        if (p_has)
                            bulk_load(sSFP + stage * C::SFP_BYTES, sfp + kb * C::SF_CHUNKS * 512, C::SFP_BYTES,
                                      sfull + stage);
                        for (int c = 0; c < 2; ++c)
                            if (qc0 + c < q_chunks_total)
                                bulk_load(sSFQ + stage * C::SFQ_BYTES + c * C::SF_CHUNKS * 512,
                                          g.q_scales + ((qc0 + c) * ksfc + kb * C::SF_CHUNKS) * 512,
                                          C::SF_CHUNKS * 512, sfull + stage);
                        issued |= 1u << stage;
                        issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                    } else {
                        if (!mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag)) {
                            ok = false;
                            break;
                        }
                        // the even CTA expects both CTAs' bytes of this operand
                        if (leader) mbar_arrive_expect_tx(full + stage, 2 * (is_p ? C::P_BYTES : C::Q_BYTES));
                        if (is_p)
                            tma_load_2d_pair(&tmP, full_leader + (uint32_t)(stage * 8), sP + stage * C::P_BYTES,
                                             (int32_t)(kb * 128), (int32_t)p_row0);
                        else
                            tma_load_2d_pair(&tmQ, full_leader + (uint32_t)(stage * 8), sQ + stage * C::Q_BYTES,
                                             (int32_t)(kb * 128), (int32_t)q_row0);
                    }
                    if (++stage == nst) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let copies already in flight land before the CTA exits.  The
                // scale copies count on this CTA's own barriers; the operand
                // copies on the even CTA's, so those get a fixed 1 ms.
                if (is_sf) {
                    WaitCfg w2 = wc;
                    if (w2.limit_ns > 1000000ull) w2.limit_ns = 1000000ull;
                    volatile int never = 0;
                    for (int s = 0; s < nst; ++s)
                        if ((issued >> s) & 1u) mbar_wait(sfull + s, (issued_ph >> s) & 1u, w2, &never);
                } else {
                    spin_ns(1000000ull);
                }
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
                    if (!mbar_wait_cluster(full + stage, ph, wc, abort_flag)) {
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
                // Wait for the tensor-core ops already issued before TMEM is freed.
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
            if (!mbar_wait(accf, aph, wc, abort_flag)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)c_begin;
            const float alpha = MX ? 1.0f : __fmul_rn(g.p_global[0], g.q_global[0]);
            uint32_t pk[NLD][16];
            // two chunks per tcgen05.wait::ld (the next tile's MMAs wait for the release)
#pragma unroll
            for (int j = 0; j < NLD; j += 2) {
                uint32_t r0[32], r1[32];
                tmem_ld32(tb + j * 32, r0);
                if (j + 1 < NLD) tmem_ld32(tb + (j + 1) * 32, r1);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[j][i] = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r0[2 * i])),
                                           __fmul_rn(alpha, __uint_as_float(r0[2 * i + 1])));
                if (j + 1 < NLD) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[j + 1][i] = pack_bf16x2(__fmul_rn(alpha, __uint_as_float(r1[2 * i])),
                                                   __fmul_rn(alpha, __uint_as_float(r1[2 * i + 1])));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader);
            aph ^= 1u;
            const int64_t pm = u % n_pm, qt = u / n_pm;
            epi_store_bf16<NLD, C::BOXC>(&tmO, smem_u32(sStg) + (uint32_t)(wg * epi_buffer_bytes<C::BOXC>()), pk, qd,
                                         lane, 1u + (uint32_t)wg, qt * BN + c_begin, pm * 256 + 128 * rank,
                                         g.q_rows_valid, g.p_rows_valid, store_pending);
        }
        if (store_pending) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the pair's MMAs, copies and TMEM reads are done in both CTAs
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace fp4
