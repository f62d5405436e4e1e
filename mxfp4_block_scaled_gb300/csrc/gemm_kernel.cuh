// gemm_kernel.cuh -- persistent block-scaled FP4 GEMM on tcgen05 (sm_103a).
//
// D[p][q] = sum_k deq(P)[p][k] * deq(Q)[q][k] for two K-major FP4 operands
// with per-16 (NVFP4, UE4M3) or per-32 (MXFP4, UE8M0) block scales, the GEMM
// of "vLLM on DGX Spark: technical report", section 6.1 (value = element x
// block scale x global scale; the global scales leave as one alpha factor).
//
// One CTA per SM, 16 warps in four warpgroups:
//   warps 0-3   scale writers: one per TMEM lane quarter; per K block they read
//               the scale atoms from smem and store them into the stage's TMEM
//               scale columns (tcgen05.st, the layout the block-scaled MMA
//               reads), so the tensor pipe is left to the MMAs.
//   warps 4, 6  TMA producers: per 256-element K block, warp 4 loads a 128-row
//               P tile and warp 6 a BN-row Q tile (128-byte swizzle).
//   warp 7      scale producer: the K block's P and Q scale atoms (plain bulk
//               copies; the MMA layout makes them contiguous) into a scale ring
//               with barriers of its own.  The writers need only those atoms
//               and the stage's TMEM columns free (the MMA's commit of the
//               previous round), so the scales are in TMEM before the operand
//               tiles land and the scale path stays off the critical path.
//   warp 5      TMEM allocator and MMA issuer (one thread): four
//               M=128 x N=BN x K=64 block-scaled MMAs per K block.
//   warps 8-15  epilogue: tcgen05.ld of the fp32 accumulator into registers,
//               release of the TMEM stage, then alpha, bf16 (or the fused MoE
//               epilogues) and global stores.  The bf16 output goes through a
//               small smem staging area (two boxes per epilogue warpgroup) and
//               TMA tensor stores, so whole lines leave the SM (row-per-thread
//               stores from registers would scatter 16-byte pieces over 32
//               lines per instruction and load the L2 with several times as
//               many write requests).
// Pipelines: STAGES operand stages (full / empty; a stage is full once both
// operand tiles landed and the four scale writers stored its scales in TMEM,
// so the MMA thread waits once per K block), as many scale slots (scale-full /
// scale-empty for the smem ring) and 1, 2 or 4 TMEM accumulator stages
// (acc_full / acc_empty; one at BN = 256).  Every wait is bounded.
// Units: tiles over a grid stride, P tiles fastest for the dense GEMM, an
// expert's weight tiles fastest for the grouped ones; the opt-in MC variant
// runs the dense kernel in clusters of two sharing each Q tile (see below).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace fp4 {

// Operand formats of the GEMM template (FK):
//   FK_NV4  NVFP4: packed E2M1 pairs, UE4M3 scale per 16 elements, alpha from
//           the two global scales (kind::mxf4nvf4, scale_vec::4X)
//   FK_MX4  MXFP4: packed E2M1 pairs, UE8M0 scale per 32 (kind::mxf4nvf4, 2X)
//   FK_MX8  MXFP8 / MXFP6: one element per byte (E4M3, E5M2, E2M3, E3M2, the
//           types named at run time in the instruction descriptor), UE8M0
//           scale per 32 (kind::mxf8f6f4, scale_vec::1X)
// The MX formats have no global scale (alpha = 1).
enum : int { FK_NV4 = 0, FK_MX4 = 1, FK_MX8 = 2 };

template <int FK>
constexpr bool fk_ue8m0() {
    return FK != FK_NV4;
}
// K elements per byte of a code row
template <int FK>
constexpr int fk_elems_per_byte() {
    return FK == FK_MX8 ? 1 : 2;
}

// bf16 epilogue staging: one buffer per epilogue warpgroup of 128 rows x
// epi_box_cols bf16 columns, the box of the output tensor map (rows of 32 or
// 64 bytes with the swizzle of that width).  Narrow boxes keep the staging
// small enough for four operand stages and a scale ring of four slots
// (NVFP4 scale slots are twice the MX ones).
template <int FK>
constexpr int epi_box_cols() {
    return FK == FK_NV4 ? 16 : 32;
}

template <int BOXC>
constexpr int epi_buffer_bytes() {
    return 128 * BOXC * 2;
}

// EPI_SWIGLU_T: the gate halves handed to the up warps, per unit parity and
// warp pair, 32 rows x 32 columns of fp32.
constexpr int kSwigluXBytes = 2 * 2 * 32 * 32 * 4;

template <int EPI>
constexpr bool epi_swapped_grouped() {
    return EPI == EPI_SWIGLU_T || EPI == EPI_DSLOT_T;
}

template <int EPI>
constexpr bool epi_grouped() {
    return EPI == EPI_SWIGLU || EPI == EPI_DSLOT || epi_swapped_grouped<EPI>();
}

// Grouped GEMMs: a CTA's first kUnitTable units' (expert, end of real token
// rows), read once after the dependency wait; the roles look them up in
// shared memory instead of each waiting on global loads per unit.
constexpr int kUnitTable = 64;
constexpr int kUnitTableBytes = kUnitTable * 8;

// EPI_DSLOT: each epilogue warp turns its 32 rows x 32 columns of fp32 around
// through 4 KB of shared memory, so that its stores cover whole rows.
constexpr int kDslotXBytes = 8 * 32 * 32 * 4;

// EPI_SWIGLU: each epilogue warp turns its 32 rows x 32 h columns (bf16)
// around through 2 KB of shared memory, so that its stores cover whole
// 64-byte row pieces.
constexpr int kSwigluStgBytes = 8 * 32 * 32 * 2;

template <int EPI, int FK>
constexpr int epi_staging_bytes() {
    return (EPI == EPI_BF16       ? 2 * epi_buffer_bytes<epi_box_cols<FK>()>()
            : EPI == EPI_SWIGLU_T ? kSwigluXBytes
            : EPI == EPI_DSLOT    ? kDslotXBytes
            : EPI == EPI_SWIGLU   ? kSwigluStgBytes
                                  : 0) +
           (epi_grouped<EPI>() ? kUnitTableBytes : 0);
}

template <int BN, int FK, int STG = 0>
struct GemmCfg {
    static constexpr int BM = 128;
    static constexpr int KB_BYTES = GEMM_KB_BYTES;                     // code bytes per row per K block
    static constexpr int KB_ELEMS = KB_BYTES * fk_elems_per_byte<FK>();  // K elements per K block
    static constexpr int KB_MMAS = KB_BYTES / 32;  // MMAs per K block (32 bytes of K each: K=64 fp4, K=32 8-bit)
    static constexpr int SF_BLOCK = FK == FK_NV4 ? 16 : 32;        // elements per block scale
    static constexpr int SF_CHUNKS = KB_ELEMS / SF_BLOCK / 4;      // 512-byte scale atoms per 128 rows per K block
    static constexpr int QCH = BN > 128 ? BN / 128 : 1;
    static constexpr int P_BYTES = BM * KB_BYTES;
    static constexpr int Q_BYTES = BN * KB_BYTES;
    static constexpr int SFP_BYTES = SF_CHUNKS * 512;
    static constexpr int SFQ_BYTES = SF_CHUNKS * 512 * QCH;
    static constexpr int OP_BYTES = P_BYTES + Q_BYTES;     // operand stage
    static constexpr int SF_BYTES = SFP_BYTES + SFQ_BYTES;  // scale slot
    // TMEM accumulator stages: the MMAs run up to ACC - 1 units ahead of the
    // epilogue (four at BN = 32, where a unit's K loop can be shorter than its
    // epilogue: the grouped GEMM2 with K = 768)
    static constexpr int ACC = BN <= 32 ? 4 : BN <= 128 ? 2 : 1;
    static constexpr int SFP_COLS = SF_CHUNKS * 4;
    static constexpr int SFQ_COLS = SF_CHUNKS * 4 * QCH;
    static constexpr int SF_COLS = SFP_COLS + SFQ_COLS;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int BUDGET = SMEM_LIMIT - 2048 - BAR_BYTES - STG;
    // operand stages (each with its TMEM scale columns), keeping room for at
    // least two scale slots; the scale ring takes what is left, up to STAGES
    static constexpr int ST_SMEM = (BUDGET - 2 * SF_BYTES) / OP_BYTES;
    static constexpr int ST_TMEM = (512 - ACC * BN) / SF_COLS;
    static constexpr int ST_MIN = ST_SMEM < ST_TMEM ? ST_SMEM : ST_TMEM;
    static constexpr int STAGES = ST_MIN < 8 ? ST_MIN : 8;
    static constexpr int SS_FIT = (BUDGET - STAGES * OP_BYTES) / SF_BYTES;
    static constexpr int SSLOTS = SS_FIT < STAGES ? SS_FIT : STAGES;
    static constexpr int STG_OFFSET =
        (STAGES * OP_BYTES + SSLOTS * SF_BYTES + 1023) / 1024 * 1024;  // swizzle alignment of the staging
    static constexpr int SMEM = 1024 + STG_OFFSET + STG + BAR_BYTES;
    static_assert(STAGES >= 2 && SSLOTS >= 2, "pipeline too shallow");
    static_assert(P_BYTES % 512 == 0 && Q_BYTES % 512 == 0, "64-byte swizzle atoms are 512 bytes");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
    static_assert(2 * STAGES + 2 * SSLOTS + 2 * ACC + 1 <= BAR_BYTES / 8 - 2, "barrier area too small");
    static_assert(ACC * BN + STAGES * SF_COLS <= 512, "TMEM budget");
};

// Work unit -> tile coordinates.
struct Unit {
    int64_t pt, qt;   // P tile, Q tile (within the expert when grouped); swapped grouped: token tile, weight tile
    int s;            // split index
    int e;            // expert (grouped) or 0
    int64_t p_row0;   // first P row
    int64_t q_row0;   // first Q row in the Q tensor
    int64_t kb0, kb1; // K-block range
    bool empty;       // swapped grouped: the token sub-tile holds no token (every role skips it)
    int64_t vend;     // grouped: end of the real rows of the unit's 128-row token tile
};

struct Sched {
    int64_t n_ptiles, n_qtiles, units, kbt, kb_per;
    int splits;
};

// Swapped grouped schedule: units = (128 / BN) sub-tiles x token tiles x the
// expert's weight tiles, weight tile fastest (the CTAs that share a token
// sub-tile run together and find it in L2) and sub-tile slowest: with a few
// tokens per expert the later sub-tiles are empty, so the units with work come
// first and the grid stride spreads them evenly over the CTAs.
// MC (CTA pairs sharing the Q tile, dense only): the P tiles go in pairs, so
// n_ptiles counts pairs of 128-row tiles (the launch makes the count even).
template <int BN, int EPI, int KB_ELEMS, bool MC = false>
__device__ __forceinline__ Sched make_sched(const GemmLaunch& g) {
    Sched s;
    s.kbt = (g.k + KB_ELEMS - 1) / KB_ELEMS;
    s.splits = g.splits;
    s.kb_per = (s.kbt + g.splits - 1) / g.splits;
    if constexpr (epi_swapped_grouped<EPI>()) {
        s.n_ptiles = (int64_t)g.n_ptiles_dev[0];  // token tiles
        s.n_qtiles = g.p_rows_valid / 128;         // weight tiles per expert
        // sub-tiles per token tile: no tile holds more than n_ptiles_dev[1]
        const int64_t subs = min((int64_t)(128 / BN), max((int64_t)1, (int64_t)g.n_ptiles_dev[1]));
        s.units = s.n_ptiles * subs * s.n_qtiles;
    } else {
        s.n_ptiles = epi_grouped<EPI>() ? (int64_t)(*g.n_ptiles_dev) : (g.p_rows_valid + 127) / 128;
        if (MC) s.n_ptiles /= 2;
        s.n_qtiles = (g.q_rows_valid + BN - 1) / BN;
        s.units = s.n_ptiles * s.n_qtiles * g.splits;
    }
    return s;
}

// The expert and real-row end of token tile pt: from the CTA's unit table
// when unit u is among its first kUnitTable, else from global memory.
__device__ __forceinline__ void unit_tile_info(const GemmLaunch& g, const int32_t* ut, int64_t u, int64_t pt,
                                               int& e, int64_t& vend) {
    const uint32_t j = (uint32_t)(u - blockIdx.x) / gridDim.x;
    if (ut && j < (uint32_t)kUnitTable) {
        e = ut[2 * j];
        vend = ut[2 * j + 1];
    } else {
        e = g.tile_expert[pt];
        vend = g.row_valid_end[pt];
    }
}

template <int BN, int EPI, bool MC = false>
__device__ __forceinline__ Unit decode_unit(const GemmLaunch& g, const Sched& sc, int64_t u,
                                            const int32_t* ut = nullptr, uint32_t prank = 0) {
    Unit w;
    w.empty = false;
    w.vend = 0;
    if constexpr (epi_swapped_grouped<EPI>()) {
        w.s = 0;
        w.qt = u % sc.n_qtiles;
        const int64_t r = u / sc.n_qtiles;
        w.pt = r % sc.n_ptiles;
        const int sub = (int)(r / sc.n_ptiles);
        unit_tile_info(g, ut, u, w.pt, w.e, w.vend);
        w.q_row0 = w.pt * 128 + sub * BN;
        w.p_row0 = (int64_t)w.e * g.p_rows_valid + w.qt * 128;
        w.kb0 = 0;
        w.kb1 = sc.kbt;
        w.empty = w.q_row0 >= w.vend;
        return w;
    }
    w.s = (int)(u % sc.splits);
    const int64_t r = u / sc.splits;
    if constexpr (epi_grouped<EPI>()) {
        // grouped: the expert's weight tiles fastest, so the units of one token
        // tile run side by side and an expert's weight tiles serve its token
        // tiles close together (token tiles fastest sent every expert's tile
        // qt to the HBM at once: the MoE call at T = 4096 took 298 against 288 us)
        w.qt = r % sc.n_qtiles;
        w.pt = r / sc.n_qtiles;
    } else {
        w.pt = r % sc.n_ptiles;
        w.qt = r / sc.n_ptiles;
    }
    if (MC) w.pt = 2 * w.pt + prank;  // the pair's tile of this CTA
    w.e = 0;
    if constexpr (epi_grouped<EPI>()) unit_tile_info(g, ut, u, w.pt, w.e, w.vend);
    w.p_row0 = w.pt * 128;
    w.q_row0 = (epi_grouped<EPI>() ? (int64_t)w.e * g.q_rows_valid : 0) + w.qt * BN;
    w.kb0 = (int64_t)w.s * sc.kb_per;
    w.kb1 = w.kb0 + sc.kb_per < sc.kbt ? w.kb0 + sc.kb_per : sc.kbt;
    return w;
}

// SiLU(g) = g / (1 + e^-g), for every element of h in the GEMM1 epilogue (h is
// requantised to FP4 right after).  e^-g = 2^(-g log2 e): the product is
// carried as p + q, p = fl(-g L) with L = fl(log2 e), q = its rounding error
// (an FMA) plus -g (log2 e - L) (Cody and Waite's split of the constant);
// 2^p comes from the hardware's ex2.approx and 2^q is 1 + q ln 2 to well
// below an ulp (|q| < 2^-16).  Then the hardware's rcp.approx and the
// product with g.  Relative error about 2^-21 (the two approximate
// instructions within about 2 ulp each, three roundings), inside the 2^-20
// the SwiGLU product is given.  For g below about -88, e^-g is +inf, the
// reciprocal 0 and SiLU 0 (the exact value is below 1e-36 in magnitude).
__device__ __forceinline__ float silu_f32(float g) {
    const float kLog2e = 1.44269502163f;        // fl(log2 e)
    const float kLog2eRest = 1.925963e-08f;      // log2 e - fl(log2 e)
    const float kLn2 = 0.693147181f;
    const float p = __fmul_rn(-g, kLog2e);
    const float q = __fadd_rn(__fmaf_rn(-g, kLog2e, -p), __fmul_rn(-g, kLog2eRest));
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(p));
    e = __fmul_rn(e, __fmaf_rn(q, kLn2, 1.0f));
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.0f, e)));
    return __fmul_rn(g, r);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Stores one epilogue warpgroup's 128 rows x (32 NLD) bf16 columns through its
// staging buffer `buf` (smem address, 1024-byte aligned) with TMA stores of
// 128 x BOXC boxes at (col0 + BOXC h, row0).  Thread (qd, lane) holds row
// 32 qd + lane; pk[j] = its columns [32 j, 32 j + 32) as packed bf16 pairs.
// A box row is BOXC * 2 bytes (32, 64 or 128) in the swizzle of that width:
// 16-byte piece c of row r sits at piece c ^ (r % 8) (128-byte rows),
// c ^ ((r / 2) % 4) (64-byte rows) or c ^ ((r / 4) % 2) (32-byte rows), which
// also keeps each st.shared free of bank conflicts.  Named barrier `bar_id` spans the warpgroup; `pending` is the
// issuing thread's record of a committed store whose smem reads may be in
// flight.
template <int NLD, int BOXC>
__device__ __forceinline__ void epi_store_bf16(const CUtensorMap* tmO, uint32_t buf, const uint32_t (&pk)[NLD][16],
                                               int qd, int lane, uint32_t bar_id, int64_t col0, int64_t row0,
                                               int64_t cols_valid, int64_t rows_valid, bool& pending) {
    static_assert(BOXC == 16 || BOXC == 32 || BOXC == 64, "32-, 64- or 128-byte box rows");
    static_assert((NLD * 32) % BOXC == 0, "whole boxes");
    constexpr int RB = BOXC * 2;   // bytes per box row
    constexpr int PIECES = RB / 16;
    const bool issuer = qd == 0 && lane == 0;
    const uint32_t r = (uint32_t)(qd * 32 + lane);
    const uint32_t row_addr = buf + r * (uint32_t)RB;
    const uint32_t sw = RB == 128 ? (r & 7u) : RB == 64 ? ((r >> 1) & 3u) : ((r >> 2) & 1u);
#pragma unroll
    for (int h = 0; h < NLD * 32 / BOXC; ++h) {
        if (issuer && pending) bulk_wait_read_all();
        named_bar_sync(bar_id, 128);  // the buffer is free
#pragma unroll
        for (int c = 0; c < PIECES; ++c) {
            const int col = h * BOXC + c * 8;  // first of the piece's 8 columns
            const int j = col / 32, i = (col % 32) / 2;
            sts128(row_addr + (((uint32_t)c ^ sw) << 4), pk[j][i], pk[j][i + 1], pk[j][i + 2], pk[j][i + 3]);
        }
        fence_proxy_async();          // generic-proxy writes -> visible to the TMA
        named_bar_sync(bar_id, 128);  // the box is complete
        if (issuer) {
            const int64_t c0 = col0 + BOXC * h;
            if (c0 < cols_valid && row0 < rows_valid) tma_store_2d(tmO, buf, (int32_t)c0, (int32_t)row0);
            bulk_commit();
            pending = true;
        }
    }
}

// Word i of the result is word (i + s) % 4 of v.
__device__ __forceinline__ uint4 rotate_words(uint4 v, uint32_t s) {
    if (s == 1) return make_uint4(v.y, v.z, v.w, v.x);
    if (s == 2) return make_uint4(v.z, v.w, v.x, v.y);
    if (s == 3) return make_uint4(v.w, v.x, v.y, v.z);
    return v;
}

// MC: clusters of two CTAs that take the two 128-row P tiles of a pair with
// the same Q tile; each CTA loads one half of the Q tile with a TMA multicast
// into both CTAs' stage (tmQ's box is BN / 2 rows), and each CTA's MMA commit
// frees the stage in both (`empty` counts the two), so a stage is rewritten
// only when both CTAs are done with it.  The L2 sends each Q tile out once
// per pair: per K block a CTA draws 16 KB of P, 16 KB of Q and its scale atoms
// from the L2 instead of 16 + 32 KB.
template <int BN, int FK, int EPI, bool MC = false>
__global__ void __launch_bounds__(512, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmO, const GemmLaunch g, const WaitCfg wc) {
    using C = GemmCfg<BN, FK, epi_staging_bytes<EPI, FK>()>;
    constexpr bool MX = fk_ue8m0<FK>();  // no global scales
    static_assert(EPI != EPI_BF16 || BN >= 128, "the staged bf16 epilogue stores 64-column boxes");
    static_assert(!MC || (EPI == EPI_BF16 && BN == 256), "CTA pairs: dense bf16 epilogue, 256-wide tiles");
    // units: a CTA takes every ustep-th unit from ucta on; a pair takes the
    // same units, each CTA its tile (prank) of the unit's pair of P tiles
    const uint32_t prank = MC ? cluster_ctarank() : 0u;
    const int64_t ucta = MC ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
    const int64_t ustep = MC ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sP = smem;
    uint8_t* sQ = sP + C::STAGES * C::P_BYTES;
    uint8_t* sSFP = sQ + C::STAGES * C::Q_BYTES;       // scale ring (SSLOTS slots)
    uint8_t* sSFQ = sSFP + C::SSLOTS * C::SFP_BYTES;
    uint8_t* sStg = smem + C::STG_OFFSET;  // bf16 epilogue staging (EPI_BF16)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + epi_staging_bytes<EPI, FK>());
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* sfull = bars + 2 * C::STAGES;                // scale atoms of the slot landed in smem
    uint64_t* sempty = sfull + C::SSLOTS;                  // the writers are done with the slot's smem
    uint64_t* accf = sempty + C::SSLOTS;
    uint64_t* acce = accf + C::ACC;
    uint64_t* drain = acce + C::ACC;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + s, 6);  // two operand producers + four scale writers
            mbar_init(empty + s, MC ? 2 : 1);  // the MMA commit (of each CTA of a pair)
        }
        for (int s = 0; s < C::SSLOTS; ++s) {
            mbar_init(sfull + s, 1);
            mbar_init(sempty + s, 4);
        }
        for (int a = 0; a < C::ACC; ++a) {
            mbar_init(accf + a, 1);
            mbar_init(acce + a, 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmP);
        prefetch_tensormap(&tmQ);
        if (EPI == EPI_BF16) prefetch_tensormap(&tmO);
    }
    if (warp == 5) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    // a pair's barriers are initialised before either CTA's copies or commits
    // can reach the other
    if (MC)
        cluster_sync();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the next kernel may be scheduled now: it waits for this grid's completion
    // before reading anything this grid writes
    pdl_launch_dependents();

    // Programmatic dependent launch: a grouped GEMM's schedule comes from the
    // preceding kernels, so every role waits here; otherwise each role waits
    // just before its first read of their outputs (the weight producer not at
    // all when early_p / early_q marks its operand).
    if (g.grouped) pdl_wait();
    const Sched sc = make_sched<BN, EPI, C::KB_ELEMS, MC>(g);
    const int32_t* ut = nullptr;  // grouped: this CTA's unit table (expert, real-row end)
    if constexpr (epi_grouped<EPI>()) {
        int32_t* t = reinterpret_cast<int32_t*>(sStg + epi_staging_bytes<EPI, FK>() - kUnitTableBytes);
        for (int j = threadIdx.x; j < kUnitTable; j += blockDim.x) {
            const int64_t u = blockIdx.x + (int64_t)j * gridDim.x;
            int32_t e = 0, vend = 0;
            if (u < sc.units) {
                int64_t pt;
                if constexpr (epi_swapped_grouped<EPI>())
                    pt = (u / sc.n_qtiles) % sc.n_ptiles;
                else
                    pt = (u / sc.splits) / sc.n_qtiles;
                e = g.tile_expert[pt];
                vend = g.row_valid_end[pt];
            }
            t[2 * j] = e;
            t[2 * j + 1] = vend;
        }
        __syncthreads();
        ut = t;
    }
    const int64_t ksfc = (g.k + 255) / 256 * (MX ? 2 : 4);      // scale atoms per 128-row tile (K padded to 256)
    static_assert(FK != FK_MX8 || C::SF_CHUNKS == 1, "an 8-bit K block is one scale atom (K padded to 256 keeps it whole)");
    const int64_t q_chunks_total = (g.q_rows + 127) / 128;      // 128-row scale tiles of Q

    if (warp < 4) {
        // ---------------------------------------------------- scale writers (smem -> TMEM only)
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int stage = 0, slot = 0;  // operand stage (TMEM scale columns), scale ring slot
        uint32_t ph = 0, sph = 0;
        for (int64_t u = ucta; u < sc.units; u += ustep) {
            const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
            if (w.empty) continue;
            // A Q tile narrower than 128 rows uses 32-row group(s) q_sub.. of each
            // scale atom; the words are rotated so those groups sit at column 0
            // of the atom's four TMEM columns: the MMA always reads the scale
            // columns from the atom's first (an offset start column at N = 32
            // faulted with a misaligned address).
            const uint32_t q_sub = BN < 128 ? (uint32_t)((w.q_row0 & 127) >> 5) : 0u;
            bool ok = true;
            for (int64_t kb = w.kb0; kb < w.kb1; ++kb) {
                // the slot's atoms are in smem, and the MMAs of the stage's
                // previous round (which read these TMEM columns) are complete
                if (!mbar_wait(sfull + slot, sph, wc, abort_flag) || !mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sfp_t = tmem + lane_base + (uint32_t)(C::ACC * BN + stage * C::SF_COLS);
                const uint32_t sfq_t = sfp_t + C::SFP_COLS;
                const uint32_t sp = smem_u32(sSFP + slot * C::SFP_BYTES) + lane * 16;
                const uint32_t sq = smem_u32(sSFQ + slot * C::SFQ_BYTES) + lane * 16;
                // lane i holds rows i, 32+i, 64+i, 96+i of an atom: TMEM lane i
                // of this quarter, columns +0..+3 (every quarter gets the atom)
#pragma unroll
                for (int c = 0; c < C::SF_CHUNKS; ++c) tmem_st4(sfp_t + c * 4, lds128(sp + c * 512));
#pragma unroll
                for (int rc = 0; rc < C::QCH; ++rc)
#pragma unroll
                    for (int c = 0; c < C::SF_CHUNKS; ++c)
                        tmem_st4(sfq_t + (c * C::QCH + rc) * 4,
                                 rotate_words(lds128(sq + (rc * C::SF_CHUNKS + c) * 512), q_sub));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(full + stage);
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
            if (!ok) break;
        }
    } else if (warp == 4 || warp == 6 || warp == 7) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producers
            // warp 4 loads the P tile, warp 6 the Q tile (each adds its own
            // bytes to the stage's barrier), warp 7 both tiles' scale atoms into
            // the scale ring; three threads issue copies in parallel.
            const bool is_p = warp == 4, is_sf = warp == 7;
            if (is_sf || (is_p ? !g.early_p : !g.early_q)) pdl_wait();
            uint64_t* const fb = is_sf ? sfull : full;   // barrier the copies complete on
            uint64_t* const eb = is_sf ? sempty : empty; // barrier that frees the slot
            const int nst = is_sf ? C::SSLOTS : C::STAGES; // ring length (stage = scale slot for warp 7)
            int stage = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, issued_ph = 0;  // per-stage bits: a copy was issued / its phase parity
            bool ok = true;
            for (int64_t u = ucta; u < sc.units && ok; u += ustep) {
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                if (w.empty) continue;
                const uint8_t* sfp = g.p_scales + (w.p_row0 >> 7) * ksfc * 512;
                const int64_t qc0 = w.q_row0 >> 7;
                for (int64_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(eb + stage, ph ^ 1u, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (is_sf) {
                        uint32_t bytes = C::SFP_BYTES;
                        for (int c = 0; c < C::QCH; ++c)
                            if (qc0 + c < q_chunks_total) bytes += C::SF_CHUNKS * 512;
                        mbar_arrive_expect_tx(sfull + stage, bytes);
                        bulk_load(sSFP + stage * C::SFP_BYTES, sfp + kb * C::SF_CHUNKS * 512, C::SFP_BYTES,
                                  sfull + stage);
                        for (int c = 0; c < C::QCH; ++c)
                            if (qc0 + c < q_chunks_total)
                                bulk_load(sSFQ + stage * C::SFQ_BYTES + c * C::SF_CHUNKS * 512,
                                          g.q_scales + ((qc0 + c) * ksfc + kb * C::SF_CHUNKS) * 512,
                                          C::SF_CHUNKS * 512, sfull + stage);
                    } else if (is_p) {
                        mbar_arrive_expect_tx(full + stage, C::P_BYTES);
                        tma_load_2d(&tmP, full + stage, sP + stage * C::P_BYTES, (int32_t)(kb * C::KB_BYTES),
                                    (int32_t)w.p_row0);
                    } else if (MC) {
                        // this CTA's half of the Q tile into both CTAs' stage; the
                        // other half comes from the other CTA
                        mbar_arrive_expect_tx(full + stage, C::Q_BYTES);
                        tma_load_2d_mc(&tmQ, full + stage, sQ + stage * C::Q_BYTES + prank * (C::Q_BYTES / 2),
                                       (int32_t)(kb * C::KB_BYTES), (int32_t)(w.q_row0 + prank * (BN / 2)),
                                       (uint16_t)3);
                    } else {
                        mbar_arrive_expect_tx(full + stage, C::Q_BYTES);
                        tma_load_2d(&tmQ, full + stage, sQ + stage * C::Q_BYTES, (int32_t)(kb * C::KB_BYTES),
                                    (int32_t)w.q_row0);
                    }
                    issued |= 1u << stage;
                    issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == nst) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let every copy already in flight land before the CTA exits.
                // Copies in flight land within microseconds; an operand stage's
                // phase may also lack the scale writers' arrivals (they stop
                // too), so each of these waits is cut short at 1 ms.
                WaitCfg w2 = wc;
                if (w2.limit_ns > 1000000ull) w2.limit_ns = 1000000ull;
                volatile int never = 0;
                for (int s = 0; s < nst; ++s)
                    if ((issued >> s) & 1u) mbar_wait(fb + s, (issued_ph >> s) & 1u, w2, &never);
                // a pair: the other CTA's multicast halves may still be landing
                // here (this CTA's barriers count them only with its own half)
                if (MC) spin_ns(200000);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc =
                FK == FK_MX8 ? idesc_mxf8f6f4(128, BN, (uint32_t)g.p_type, (uint32_t)g.q_type) : idesc_mxf4(128, BN, MX);
            int stage = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t aph = 0;
            bool ok = true, any = false;
            for (int64_t u = ucta; u < sc.units && ok; u += ustep) {
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                if (w.empty) continue;
                if (!mbar_wait(acce + acc, aph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                for (int64_t kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(full + stage, ph, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfp_t = tmem + (uint32_t)(C::ACC * BN + stage * C::SF_COLS);
                    const uint32_t sfq_t = sfp_t + C::SFP_COLS;
                    const uint32_t pa = smem_u32(sP + stage * C::P_BYTES);
                    const uint32_t qa = smem_u32(sQ + stage * C::Q_BYTES);
#pragma unroll
                    for (int kk = 0; kk < C::KB_MMAS; ++kk) {
                        const uint64_t ad = C::KB_BYTES == 128 ? sdesc_sw128(pa + kk * 32) : sdesc_sw64(pa + kk * 32);
                        const uint64_t bd = C::KB_BYTES == 128 ? sdesc_sw128(qa + kk * 32) : sdesc_sw64(qa + kk * 32);
                        uint32_t sfa, sfb, id;
                        if constexpr (FK == FK_NV4) {
                            sfa = sfp_t + kk * 4;
                            sfb = sfq_t + kk * 4 * C::QCH;
                            id = idesc;
                        } else if constexpr (FK == FK_MX4) {
                            sfa = sfp_t + (kk >> 1) * 4;
                            sfb = sfq_t + (kk >> 1) * 4 * C::QCH;
                            id = idesc_with_sf_id(idesc, (uint32_t)(kk & 1) * 2u);
                        } else {
                            // one scale byte per row per K=32 MMA: byte kk of the atom's word
                            sfa = sfp_t;
                            sfb = sfq_t;
                            id = idesc_with_sf_id(idesc, (uint32_t)kk);
                        }
                        const uint32_t acc_in = (kb > w.kb0 || kk > 0) ? 1u : 0u;
                        if constexpr (FK == FK_MX8)
                            mma_mxf8f6f4(d_tmem, ad, bd, id, sfa, sfb, acc_in);
                        else
                            mma_mxf4<MX>(d_tmem, ad, bd, id, sfa, sfb, acc_in);
                    }
                    any = true;
                    if (MC)
                        mma_commit_mc(empty + stage, (uint16_t)3);  // frees the stage in both CTAs
                    else
                        mma_commit(empty + stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf + acc);
                if (++acc == C::ACC) {
                    acc = 0;
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
    } else if (warp >= 8) {
        // ---------------------------------------------------- epilogue
        // 8 warps: warp w owns TMEM lane quarter (w % 4) and column half
        // (w - 8) / 4.  Each pulls all its accumulator columns into registers
        // (back-to-back tcgen05.ld, one wait), releases the accumulator stage
        // at once, then converts and stores while the next tile's MMAs run.
        constexpr int GRAN = EPI == EPI_SWIGLU ? 64 : epi_swapped_grouped<EPI>() ? 16 : 32;
        constexpr int CPW = BN / 2 > GRAN ? BN / 2 : GRAN;  // columns per warp
        constexpr int NLD = CPW / 32;
        static_assert(EPI != EPI_DSLOT || CPW <= 64, "fp32 rows keep their columns in registers");
        const int qd = warp & 3;  // the TMEM lane quarter this warp may access
        const int c_begin = ((warp - 8) >> 2) * CPW;
        const bool has_cols = c_begin < BN;
        const int wg = (warp - 8) >> 2;
        pdl_wait();  // global scales and output buffers
        bool store_pending = false;  // EPI_BF16: this thread issued a TMA store not yet waited for
        int acc = 0;
        uint32_t aph = 0;
        uint32_t n_done = 0;  // units converted by this warp (EPI_SWIGLU_T buffer parity)
        for (int64_t u = ucta; u < sc.units; u += ustep) {
            if constexpr (epi_swapped_grouped<EPI>()) {
                const Unit wp = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                if (wp.empty) continue;
            }
            if (!mbar_wait(accf + acc, aph, wc, abort_flag)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(acc * BN + c_begin);

            if constexpr (EPI == EPI_BF16) {
                // two chunks per round (one tcgen05.wait::ld each): fp32 -> alpha ->
                // packed bf16 pairs, then release.  The MMAs of the next tile wait
                // for the release, so its latency is paid at every tile boundary
                // (one round per chunk cost ~1,000 cycles there, 8 % of the prefill).
                const float alpha = MX ? 1.0f : __fmul_rn(g.p_global[0], g.q_global[0]);
                uint32_t pk[NLD][16];
                if (has_cols) {
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
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                constexpr int BOXC = epi_box_cols<FK>();
                epi_store_bf16<NLD, BOXC>(&tmO, smem_u32(sStg) + (uint32_t)(wg * epi_buffer_bytes<BOXC>()), pk, qd, lane,
                                    1u + (uint32_t)wg, w.qt * BN + c_begin, w.p_row0, g.q_rows_valid,
                                    g.p_rows_valid, store_pending);
            } else if constexpr (EPI == EPI_BF16_T || EPI == EPI_PARTIAL_T) {
                uint32_t r[NLD][32];
                if (has_cols) {
#pragma unroll
                    for (int j = 0; j < NLD; ++j) tmem_ld32(tb + j * 32, r[j]);
                    tmem_ld_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                const int64_t prow = w.p_row0 + qd * 32 + lane;
                const float alpha = MX ? 1.0f : __fmul_rn(g.p_global[0], g.q_global[0]);
                if (has_cols && prow < g.p_rows_valid) {
#pragma unroll
                    for (int j = 0; j < NLD; ++j) {
                        const int64_t q0 = w.qt * BN + c_begin + j * 32;  // first token of the chunk
                        if constexpr (EPI == EPI_BF16_T) {
                            uint16_t* o = reinterpret_cast<uint16_t*>(g.out);
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int64_t t = q0 + i;
                                if (t < g.q_rows_valid) {
                                    __nv_bfloat16 h =
                                        __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[j][i])));
                                    o[t * g.ldo + prow] = *reinterpret_cast<uint16_t*>(&h);
                                }
                            }
                        } else {
                            float* o = reinterpret_cast<float*>(g.out) +
                                       (int64_t)w.s * g.q_rows_valid * g.p_rows_valid;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int64_t t = q0 + i;
                                if (t < g.q_rows_valid) o[t * g.p_rows_valid + prow] = __uint_as_float(r[j][i]);
                            }
                        }
                    }
                }
            } else if constexpr (EPI == EPI_PARTIAL) {
                // split-K partials, row-major; only the warps holding real rows
                // read TMEM (for decode-sized M that is one lane quarter)
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                const int64_t row0 = w.p_row0 + qd * 32;
                const bool any_rows = has_cols && row0 < g.p_rows_valid;
                const int64_t prow = row0 + lane;
                float* o = reinterpret_cast<float*>(g.out) + ((int64_t)w.s * g.p_rows_valid + prow) * g.ldo;
                if (any_rows) {
#pragma unroll 1
                    for (int j = 0; j < NLD; ++j) {
                        uint32_t r[32];
                        tmem_ld32(tb + j * 32, r);
                        tmem_ld_wait();
                        const int64_t q0 = w.qt * BN + c_begin + j * 32;
                        if (prow < g.p_rows_valid) {
                            float4* o4 = reinterpret_cast<float4*>(o + q0);
                            if (q0 + 32 <= g.q_rows_valid) {
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    o4[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                            } else {
                                for (int i = 0; i < 32; ++i)
                                    if (q0 + i < g.q_rows_valid) o[q0 + i] = __uint_as_float(r[i]);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
            } else if constexpr (EPI == EPI_SWIGLU) {
                // Q rows are W13 rows interleaved in groups of 32 (gate, up, gate, up, ...):
                // columns [c, c+32) are gate and [c+32, c+64) up for the same 32 features.
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                const int64_t prow = w.p_row0 + qd * 32 + lane;
                const float alpha =
                    __fmul_rn(g.p_global_per_expert ? g.p_global[w.e] : g.p_global[0], g.q_global[w.e]);
                uint32_t hv[NLD / 2][16];
                uint32_t amax_bits = 0;
                if (has_cols) {
#pragma unroll
                    for (int j = 0; j < NLD; j += 2) {
                        uint32_t rg[32], ru[32];
                        tmem_ld32(tb + j * 32, rg);
                        tmem_ld32(tb + j * 32 + 32, ru);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float g0 = __fmul_rn(alpha, __uint_as_float(rg[2 * i]));
                            const float g1 = __fmul_rn(alpha, __uint_as_float(rg[2 * i + 1]));
                            const float u0 = __fmul_rn(alpha, __uint_as_float(ru[2 * i]));
                            const float u1 = __fmul_rn(alpha, __uint_as_float(ru[2 * i + 1]));
                            hv[j / 2][i] = pack_bf16x2(__fmul_rn(silu_f32(g0), u0), __fmul_rn(silu_f32(g1), u1));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
                // the amax of the row's h values (bf16 bits, sign cleared)
                if (has_cols && prow < w.vend) {
#pragma unroll
                    for (int jp = 0; jp < NLD / 2; ++jp)
#pragma unroll
                        for (int i = 0; i < 16; ++i) amax_bits = __vmaxu2(amax_bits, hv[jp][i] & 0x7FFF7FFFu);
                }
                // rows through shared memory: lane i writes row i's 64 bytes (16-byte
                // piece v at v ^ ((i / 2) % 4): the eight lanes of a store phase hit
                // distinct banks), then each store instruction covers 8 rows x 64
                // contiguous bytes
                if (has_cols) {
                    const uint32_t xs = smem_u32(sStg) + (uint32_t)(warp - 8) * 2048u;
                    const int64_t prow0 = w.p_row0 + qd * 32;
                    uint16_t* hbase = reinterpret_cast<uint16_t*>(g.out);
#pragma unroll
                    for (int jp = 0; jp < NLD / 2; ++jp) {
                        const int64_t f0 = (w.qt * BN + c_begin + jp * 64) / 2;  // first h column of the pair
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            sts128(xs + (uint32_t)lane * 64u + ((uint32_t)(v ^ ((lane >> 1) & 3)) << 4), hv[jp][4 * v],
                                   hv[jp][4 * v + 1], hv[jp][4 * v + 2], hv[jp][4 * v + 3]);
                        __syncwarp();
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = i * 8 + (lane >> 2), c4 = lane & 3;
                            const uint4 v4 = lds128(xs + (uint32_t)row * 64u + ((uint32_t)(c4 ^ ((row >> 1) & 3)) << 4));
                            if (prow0 + row < w.vend)
                                *reinterpret_cast<uint4*>(hbase + (prow0 + row) * g.ldo + f0 + c4 * 8) = v4;
                        }
                        __syncwarp();
                    }
                }
                if (has_cols) {
                    uint32_t m = max(amax_bits & 0xFFFFu, amax_bits >> 16);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                    if (lane == 0 && m) atomicMax(reinterpret_cast<unsigned int*>(g.amax_out) + w.e, m << 16);
                }
            } else if constexpr (EPI == EPI_DSLOT) {
                // token rows (expert-sorted, padded): D[row][feature] = alpha * acc
                // (fp32).  Per 32-column chunk the warp writes its 32 rows to its
                // 4 KB of shared memory in the 128-byte swizzle (row r's 16-byte
                // piece v at piece v ^ (r % 8): no bank conflicts) and one TMA store
                // takes the 32 x 32 box out; a box of padding rows only is skipped.
                uint32_t r[NLD][32];
                if (has_cols) {
#pragma unroll
                    for (int j = 0; j < NLD; ++j) tmem_ld32(tb + j * 32, r[j]);
                    tmem_ld_wait();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                const int64_t prow0 = w.p_row0 + qd * 32;
                const float alpha = __fmul_rn(g.p_global[w.e], g.q_global[w.e]);
                const uint32_t xs = smem_u32(sStg) + (uint32_t)(warp - 8) * 4096u;
                if (has_cols && prow0 < w.vend) {
#pragma unroll
                    for (int j = 0; j < NLD; ++j) {
                        if (lane == 0 && store_pending) bulk_wait_read_all();  // the buffer is free
                        __syncwarp();
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            sts128(xs + (uint32_t)lane * 128u + ((uint32_t)(v ^ (lane & 7)) << 4),
                                   __float_as_uint(__fmul_rn(alpha, __uint_as_float(r[j][4 * v]))),
                                   __float_as_uint(__fmul_rn(alpha, __uint_as_float(r[j][4 * v + 1]))),
                                   __float_as_uint(__fmul_rn(alpha, __uint_as_float(r[j][4 * v + 2]))),
                                   __float_as_uint(__fmul_rn(alpha, __uint_as_float(r[j][4 * v + 3]))));
                        fence_proxy_async();  // generic-proxy writes -> visible to the TMA
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmO, xs, (int32_t)(w.qt * BN + c_begin + j * 32), (int32_t)prow0);
                            bulk_commit();
                            store_pending = true;
                        }
                    }
                }
            } else if constexpr (EPI == EPI_DSLOT_T) {
                // P rows are the expert's W2 rows (output features), columns the
                // sub-tile's token rows (expert-sorted): d[row of column][feature] =
                // alpha * acc; the 32 lanes of a column write 32 consecutive features
                static_assert(CPW % 16 == 0, "whole 16-column loads");
                uint32_t r[CPW / 16][16];
#pragma unroll
                for (int c = 0; c < CPW / 16; ++c) tmem_ld16(tb + c * 16, r[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                const float alpha = __fmul_rn(g.q_global[w.e], g.p_global[w.e]);
                const int64_t hd = w.qt * 128 + qd * 32 + lane;
                const int64_t vend = w.vend;
                const int64_t row0 = w.q_row0 + c_begin;
                float* d = reinterpret_cast<float*>(g.out) + hd;
#pragma unroll
                for (int c = 0; c < CPW; ++c)
                    if (row0 + c < vend) d[(row0 + c) * g.ldo] = __fmul_rn(alpha, __uint_as_float(r[c / 16][c % 16]));
            } else if constexpr (EPI == EPI_SWIGLU_T) {
                // P rows are the expert's W13 rows, interleaved in groups of 32
                // (gate, up, ...): TMEM lane quarters 0 / 1 hold gate / up of
                // features 64 qt + [0, 32), quarters 2 / 3 of 64 qt + [32, 64);
                // the 32 columns are the sub-tile's token rows, 16 per warpgroup.
                // In each gate / up warp pair the gate warp converts the first 8
                // of its 16 columns and the up warp the last 8; each hands the
                // other its alpha * acc for the other's columns through smem.
                static_assert(BN == 32, "16 columns per epilogue warp");
                uint32_t r[16];
                tmem_ld16(tb, r);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + acc);
                const Unit w = decode_unit<BN, EPI, MC>(g, sc, u, ut, prank);
                const float alpha = __fmul_rn(g.q_global[g.q_global_per_expert ? w.e : 0], g.p_global[w.e]);
                const int pair = qd >> 1, half = wg;
                const bool is_gate = (qd & 1) == 0;
                // [parity][half][pair][direction][8 columns][32 lanes]
                float* xb = reinterpret_cast<float*>(sStg) + ((((n_done & 1u) * 2 + half) * 2 + pair) * 2) * 8 * 32;
                float* to_up = xb;             // gate of columns 8..15
                float* to_gate = xb + 8 * 32;  // up of columns 0..7
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (is_gate)
                        to_up[i * 32 + lane] = __fmul_rn(alpha, __uint_as_float(r[8 + i]));
                    else
                        to_gate[i * 32 + lane] = __fmul_rn(alpha, __uint_as_float(r[i]));
                }
                named_bar_sync(3u + (uint32_t)(half * 2 + pair), 64);
                const int64_t f = w.qt * 64 + pair * 32 + lane;
                const int64_t vend = w.vend;
                const int64_t row0 = w.q_row0 + c_begin + (is_gate ? 0 : 8);
                uint16_t* o = reinterpret_cast<uint16_t*>(g.out);
                uint32_t amax_bits = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float gt = is_gate ? __fmul_rn(alpha, __uint_as_float(r[i])) : to_up[i * 32 + lane];
                    const float up = is_gate ? to_gate[i * 32 + lane] : __fmul_rn(alpha, __uint_as_float(r[8 + i]));
                    const int64_t row = row0 + i;
                    if (row < vend) {
                        const __nv_bfloat16 hb = __float2bfloat16_rn(__fmul_rn(silu_f32(gt), up));
                        const uint16_t hbits = *reinterpret_cast<const uint16_t*>(&hb);
                        o[row * g.ldo + f] = hbits;
                        amax_bits = max(amax_bits, (uint32_t)(hbits & 0x7FFFu));
                    }
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o2));
                if (lane == 0 && amax_bits) atomicMax(reinterpret_cast<unsigned int*>(g.amax_out) + w.e, amax_bits << 16);
                ++n_done;
            }
            if (++acc == C::ACC) {
                acc = 0;
                aph ^= 1u;
            }
        }
        if (store_pending) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // a pair: neither CTA leaves while the other's copies or commits can
    // still reach its shared memory
    if (MC) cluster_sync();
}

}  // namespace fp4
