// moe_fused.cu -- the NVFP4 fused-MoE layer for a few tokens in ONE launch.
//
// The same computation as the launch chain of moe.cu ("vLLM on DGX Spark:
// technical report", section 7.1: route -> quantise/dispatch -> experts ->
// combine, with the expert computation of section 4.3: two GEMMs, SwiGLU and
// a top-k weighted reduction; section 4.5 describes one fused kernel that
// takes bf16 in and quantises inside), for T <= kFusedMaxT tokens: the call
// is a stream of the touched experts' weights, so every CTA starts its weight
// stream as soon as it knows the routing, and the cross-CTA dependencies go
// through counters in the workspace instead of kernel boundaries.
//
// Grid: one CTA per SM, launched cooperatively (all CTAs resident, so a CTA
// may wait for another).  Every CTA routes all T tokens itself (a warp per
// token) and takes the NVFP4 global scale of the hidden rows (dynamic: amax /
// 2688 over the whole tensor), so all CTAs agree on the active experts
// act[0..E_act) (ascending) and each expert's token slots (token order).
// Work units, taken round-robin (unit v = blockIdx.x + i * gridDim.x):
//   GEMM1 unit (a, t)  128 interleaved W13 rows of expert act[a] (64 features
//                      of gate and up), K = H: h[slot][64 t .. 64 t + 64) =
//                      bf16(SiLU(alpha1 G_gate) * alpha1 G_up), amax of h;
//                      then cnt1[a] += 1
//   GEMM2 unit (a, t)  128 W2 rows (output features 128 t ..), K = I: waits
//                      for cnt1[a] == 2I / 128, requantises the expert's h rows
//                      with s_gH = amax / 2688 (static: static2[e]),
//                      D[slot][f] = alpha2 acc; then cnt2[t] += 1, and the
//                      CTA that brings cnt2[t] to E_act sums, for every token
//                      and feature of the tile, w[t][j] D[slot(t, j)] in slot
//                      order j = 0..k-1 (fp32) and writes the bf16 output.
// Every GEMM1 unit precedes every GEMM2 unit in each CTA's list, so no CTA
// waits while holding GEMM1 work: with all CTAs resident this cannot
// deadlock.  The counters (and the amax) must be zero at launch: the host
// clears them with one memset before the kernel.
//
// Per CTA, 16 warps, the units flowing through them as a pipeline:
//   warp 4      TMA producer: each unit's weight tile per 256-element K block
//               (128 rows x 128 B, 128-byte swizzle) and its 4 scale atoms,
//               on one barrier per stage; it runs ahead through the ring
//               from the first unit (the weights depend only on the routing)
//   warps 12-15 the token operand of each unit (the hidden rows quantised
//               with the unit's global scale, or -- after the expert's GEMM1
//               units -- its h rows requantised) for the whole K into one of
//               two shared-memory tiles, so unit n + 1's operand is built
//               while unit n computes
//   warps 0-3   scale writers: the stage's weight atoms and the unit's token
//               atoms of that K block into the stage's TMEM scale columns
//   warp 5      TMEM allocation and the MMA issuer: swap-AB block-scaled MMAs
//               (M = 128 weight rows, N = 32 token columns, K = 64) into one
//               of two TMEM accumulators
//   warps 8-11  the epilogue of each unit, overlapping the next unit's MMAs
// Every wait is bounded: on expiry the role sets the device error word and
// an abort flag that stops the others in the CTA (a CTA waiting on a counter
// that an aborted CTA never raises gives up at its own limit).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "gemm_kernel.cuh"
#include "internal.h"
#include "moe_common.cuh"
#include "quant_math.cuh"

namespace fp4 {

struct FusedCfg {
    static constexpr int BN = 32;                          // token columns (an expert has at most T <= 32 tokens)
    static constexpr int P_BYTES = 128 * 128;              // weight tile per K block
    static constexpr int SFP_BYTES = 4 * 512;              // weight scale atoms per K block
    static constexpr int MAX_KB = kFusedMaxK / 256;        // K blocks of the token operand
    static constexpr int QC_BYTES = BN * 128;              // token codes per K block (32 rows x 128 B)
    // token scale atoms per K block, compact: the 32 token rows' words of the
    // four atoms (row r's 4 bytes at c * 128 + r * 4); the scale writers
    // expand them to the TMEM layout (rows 32-127 of an atom are zero)
    static constexpr int QS_BYTES = 4 * 128;
    static constexpr int QBUF = MAX_KB * (QC_BYTES + QS_BYTES);  // one token operand tile (codes, then atoms)
    static constexpr int STAGES = 7;
    static constexpr int SF_COLS = 32;                     // TMEM scale columns per stage (16 weight + 16 token)
    static constexpr int XCH_BYTES = 4 * kFusedMaxT * 32 * 4;  // the epilogue's alpha-scaled accumulator columns
    static constexpr int OFF_P = 0;
    static constexpr int OFF_SF = OFF_P + STAGES * P_BYTES;
    static constexpr int OFF_Q = OFF_SF + STAGES * SFP_BYTES;  // two token operand tiles
    static constexpr int OFF_X = OFF_Q + 2 * QBUF;
    static constexpr int OFF_DTAB = OFF_X + XCH_BYTES;     // three divisor tables: GEMM1 dynamic, per tile x 2
    static constexpr int OFF_TAB = OFF_DTAB + 3 * 128 * 8;
    // routing tables: ids and weights per slot; per expert the token mask,
    // active index and the two weight global scales; per active expert the
    // expert, its slot list, token count and s_gH; misc words
    static constexpr int TAB_BYTES = kFusedMaxSlots * 4 * 2 + kFusedMaxE * (4 + 2 + 4 + 4) +
                                     kFusedMaxSlots * (4 + kFusedMaxT * 2 + 4 + 4) + 256;
    static constexpr int OFF_BAR = OFF_TAB + TAB_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM = 1024 + OFF_BAR + BAR_BYTES;
    static_assert(OFF_Q % 1024 == 0 && QBUF % 1024 == 0 && OFF_P % 1024 == 0, "swizzled tiles are 1024-byte aligned");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(2 * BN + STAGES * SF_COLS <= 512, "TMEM budget");
    static_assert(kFusedMaxT <= BN, "an expert's tokens fit the N side");
};

struct FusedMoeArgs {
    const uint16_t* hidden;  // bf16 [T][H]
    const float* logits;     // fp32 [T][E]
    int T, H, I, E, k;
    int is_static;
    const uint8_t* w13_scales;
    const float* w13_global;  // [E]
    const uint8_t* w2_scales;
    const float* w2_global;   // [E]
    uint16_t* out;            // bf16 [T][H]
    // workspace
    int32_t* ids;             // [T k]
    float* weights;           // [T k]
    float* sg_a;              // [1] dynamic s_gA
    uint32_t* cnt1;           // [kFusedMaxSlots] zeroed
    uint32_t* cnt2;           // [kFusedMaxOutTiles] zeroed
    uint32_t* amax_h;         // [kFusedMaxSlots] zeroed (fp32 bits of |h| maxima)
    uint16_t* h;              // bf16 [T k][I], slot order
    uint8_t* a_codes;         // [T k][H/2] the dispatched hidden rows' codes, slot order
    uint8_t* a_sbytes;        // [T k][H/16] their scale bytes (row-major)
    uint8_t* h_codes;         // [T k][I/2] the requantised h rows' codes
    uint8_t* h_sbytes;        // [T k][I/16] their scale bytes
    float* sg_h;              // [E] s_gH of each active expert
    float* d;                 // fp32 [T k][H] alpha2-scaled expert outputs
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait, by one thread, for a counter another CTA raises; false (and
// the device error word and the CTA's abort flag set) when it gives up.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t want, const WaitCfg& wc,
                                           volatile int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < 0x40000000u; ++it) {
        if (ld_acquire_u32(p) >= want) return true;
        if (*abort_flag) return false;
        __nanosleep(32);
        if ((it & 15u) == 15u && globaltimer_ns() - t0 > wc.limit_ns) break;
    }
    atomicOr(wc.err, DEV_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

template <int PER_LANE>
__global__ void __launch_bounds__(512, 1)
    moe_fused_kernel(const __grid_constant__ CUtensorMap tm13, const __grid_constant__ CUtensorMap tm2,
                     const FusedMoeArgs a, const StaticScales st, const WaitCfg wc) {
    using C = FusedCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sP = smem + C::OFF_P;
    uint8_t* sSF = smem + C::OFF_SF;
    uint8_t* sQ = smem + C::OFF_Q;  // tile b: codes at b * QBUF, atoms at b * QBUF + MAX_KB * QC_BYTES
    float* sX = reinterpret_cast<float*>(smem + C::OFF_X);
    float2* dtab = reinterpret_cast<float2*>(smem + C::OFF_DTAB);  // [3][128]
    int32_t* s_ids = reinterpret_cast<int32_t*>(smem + C::OFF_TAB);
    float* s_w = reinterpret_cast<float*>(s_ids + kFusedMaxSlots);
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_w + kFusedMaxSlots);    // [E] tokens of each expert (bit t)
    float* s_gw13 = reinterpret_cast<float*>(s_mask + kFusedMaxE);           // [E] W13 global scales
    float* s_gw2 = s_gw13 + kFusedMaxE;                                      // [E] W2 global scales
    int16_t* s_aidx = reinterpret_cast<int16_t*>(s_gw2 + kFusedMaxE);        // [E] active index
    int32_t* s_act = reinterpret_cast<int32_t*>(s_aidx + kFusedMaxE);        // [E_act] expert
    int16_t* s_eslot = reinterpret_cast<int16_t*>(s_act + kFusedMaxSlots);   // [E_act][kFusedMaxT] slots
    int32_t* s_ne = reinterpret_cast<int32_t*>(s_eslot + kFusedMaxSlots * kFusedMaxT);  // [E_act] token count
    float* s_sgh = reinterpret_cast<float*>(s_ne + kFusedMaxSlots);          // [E_act] s_gH (quantisers -> epilogue)
    // [0] E_act, [1] amax bits, [2] last-arriver flag, [3] the quantisers' s_g,
    // [4..36) per-chunk active counts (prologue), then [4] the quantisers' and
    // [5] the epilogue's stop flags
    volatile int32_t* s_misc = reinterpret_cast<int32_t*>(s_sgh + kFusedMaxSlots);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tready = bars + 2 * C::STAGES;
    uint64_t* qfull = bars + 3 * C::STAGES;  // [2] token tile written
    uint64_t* qempty = qfull + 2;            // [2] the MMAs reading the tile are done
    uint64_t* accf = qempty + 2;             // [2] accumulator complete
    uint64_t* acce = accf + 2;               // [2] accumulator read by the epilogue
    uint64_t* drain = acce + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, H = a.H, I = a.I, E = a.E, k = a.k;
    // The routing and the hidden abs-max need only the inputs: their loads go
    // out first (after the dependency wait), before the set-up below.
    pdl_wait();  // hidden and logits come from the preceding kernels
    float lg[PER_LANE];
    if (warp < T) {
#pragma unroll
        for (int q = 0; q < PER_LANE; ++q) {
            const int e = q * 32 + lane;
            lg[q] = e < E ? __ldg(a.logits + (int64_t)warp * E + e) : -INFINITY;
        }
    }
    const float gw = threadIdx.x < E ? __ldg(a.w13_global + threadIdx.x) : 0.0f;
    const float gw2 = threadIdx.x < E ? __ldg(a.w2_global + threadIdx.x) : 0.0f;
    uint32_t hm = 0;
    if (!a.is_static) {
        const int nv = T * H / 8;
        const uint4* xv = reinterpret_cast<const uint4*>(a.hidden);
        for (int i = threadIdx.x; i < nv; i += 512) hm = absmax8(__ldg(xv + i), hm);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
            mbar_init(tready + s, 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(qfull + b, 1);
            mbar_init(qempty + b, 1);
            mbar_init(accf + b, 1);
            mbar_init(acce + b, 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tm13);
        prefetch_tensormap(&tm2);
    }
    // the token tiles' scale words start at zero: the rows past a unit's tokens
    // (codes and scales left from set-up or an earlier unit) feed only
    // accumulator columns nobody reads, and zero or earlier finite scales keep
    // even those finite; the codes need no clearing (E2M1 codes are finite)
    for (int i = threadIdx.x; i < 2 * C::MAX_KB * C::QS_BYTES / 16; i += 512) {
        const int b = i / (C::MAX_KB * C::QS_BYTES / 16), r = i - b * (C::MAX_KB * C::QS_BYTES / 16);
        reinterpret_cast<uint4*>(sQ + b * C::QBUF + C::MAX_KB * C::QC_BYTES)[r] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (threadIdx.x < E) {
        s_mask[threadIdx.x] = 0u;
        s_gw13[threadIdx.x] = gw;
        s_gw2[threadIdx.x] = gw2;
    }
    fence_proxy_async();
    if (warp == 5) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // ---------------------------------------------------------- prologue
    // route (a warp per token, ties to the lower expert index) and the
    // hidden rows' abs-max
    if (warp < T) {
        int e;
        float w;
        topk_regs<PER_LANE>(lg, E, k, lane, e, w);
        if (lane < k) {
            s_ids[warp * k + lane] = e;
            s_w[warp * k + lane] = w;
        }
    }
    if (!a.is_static) {
        hm = max(hm & 0xFFFFu, hm >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) hm = max(hm, __shfl_xor_sync(0xFFFFFFFFu, hm, o));
        if (lane == 0) s_misc[4 + warp] = (int32_t)hm;
    }
    __syncthreads();
    if (threadIdx.x < T * k) atomicOr(&s_mask[s_ids[threadIdx.x]], 1u << (threadIdx.x / k));
    if (!a.is_static && threadIdx.x < 32) {
        uint32_t m = lane < 16 ? (uint32_t)s_misc[4 + lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) s_misc[1] = (int32_t)m;
    }
    __syncthreads();
    const float sg_a = a.is_static ? 0.0f : __fdiv_rn(__uint_as_float((uint32_t)s_misc[1] << 16), 2688.0f);
    // the GEMM1 divisor table of the dynamic scale (one for every GEMM1 unit)
    if (!a.is_static && threadIdx.x >= 384) dtab[threadIdx.x - 384] = nvfp4_divisor(threadIdx.x - 384, sg_a, T > 2);
    // active experts in ascending order: warp w ballots experts 64 w .. 64 w + 63
    uint32_t bal[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int e = warp * 64 + c * 32 + lane;
        bal[c] = __ballot_sync(0xFFFFFFFFu, e < E && s_mask[e] != 0u);
        if (lane == 0) s_misc[4 + warp * 2 + c] = __popc(bal[c]);
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive prefix over the 32 chunk counts
        const int n = s_misc[4 + lane];
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncwarp();
        s_misc[4 + lane] = incl - n;
        if (lane == 31) s_misc[0] = incl;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int e = warp * 64 + c * 32 + lane;
        if ((bal[c] >> lane) & 1u) {
            const int idx = s_misc[4 + warp * 2 + c] + __popc(bal[c] & ((1u << lane) - 1u));
            s_act[idx] = e;
            s_aidx[e] = (int16_t)idx;
            s_ne[idx] = __popc(s_mask[e]);
        }
    }
    __syncthreads();
    if (threadIdx.x < T * k) {
        const int i = threadIdx.x, t = i / k, e = s_ids[i];
        const int pos = __popc(s_mask[e] & ((1u << t) - 1u));  // the expert's tokens before t
        s_eslot[s_aidx[e] * kFusedMaxT + pos] = (int16_t)i;
        if (blockIdx.x == 0) {
            a.ids[i] = e;
            a.weights[i] = s_w[i];
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && !a.is_static) a.sg_a[0] = sg_a;
    __syncthreads();
    const int E_act = s_misc[0];
    const int n1 = 2 * I / 128, n2 = H / 128;
    const int U1 = E_act * n1, U = U1 + E_act * n2;
    const int kb1 = H / 256, kb2 = I / 256;
    const int64_t ksfc13 = (int64_t)(H / 256) * 4, ksfc2 = (int64_t)(I / 256) * 4;
    // (no early trigger of dependent launches: this grid's CTAs wait on one
    // another, so nothing else is invited onto their SMs before they finish)

    // unit v -> (GEMM1?, active index, tile)
    auto unit = [&](int v, bool& g1, int& ai, int& t) {
        g1 = v < U1;
        const int w = g1 ? v : v - U1;
        const int n = g1 ? n1 : n2;
        ai = w / n;
        t = w - ai * n;
    };

    if (warp < 4) {
        // ------------------------------------------------ scale writers
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        int n = 0;
        for (int v = blockIdx.x; v < U && ok; v += gridDim.x, ++n) {
            bool g1;
            int ai, t;
            unit(v, g1, ai, t);
            const int qb = n & 1;
            if (!mbar_wait(qfull + qb, (uint32_t)(n >> 1) & 1u, wc, abort_flag)) break;
            const int kbn = g1 ? kb1 : kb2;
            const uint32_t qs0 = smem_u32(sQ + qb * C::QBUF + C::MAX_KB * C::QC_BYTES) + lane * 4;
            for (int kb = 0; kb < kbn; ++kb) {
                if (!mbar_wait(full + stage, ph, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t sfp_t = tmem + lane_base + (uint32_t)(2 * C::BN + stage * C::SF_COLS);
                const uint32_t sfq_t = sfp_t + 16;
                const uint32_t sp = smem_u32(sSF + stage * C::SFP_BYTES) + lane * 16;
                const uint32_t sq = qs0 + kb * C::QS_BYTES;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tmem_st4(sfp_t + c * 4, lds128(sp + c * 512));
                    uint32_t wq;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(wq) : "r"(sq + c * 128));
                    tmem_st4(sfq_t + c * 4, make_uint4(wq, 0u, 0u, 0u));
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tready + stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 4) {
        if (lane == 0) {
            // ------------------------------------------------ weight producer
            int stage = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, issued_ph = 0;
            bool ok = true;
            for (int v = blockIdx.x; v < U && ok; v += gridDim.x) {
                bool g1;
                int ai, t;
                unit(v, g1, ai, t);
                const int e = s_act[ai];
                const int64_t row0 = g1 ? (int64_t)e * 2 * I + t * 128 : (int64_t)e * H + t * 128;
                const uint8_t* sf = g1 ? a.w13_scales + (row0 >> 7) * ksfc13 * 512 : a.w2_scales + (row0 >> 7) * ksfc2 * 512;
                const int kbn = g1 ? kb1 : kb2;
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full + stage, C::P_BYTES + C::SFP_BYTES);
                    tma_load_2d(g1 ? &tm13 : &tm2, full + stage, sP + stage * C::P_BYTES, kb * 128, (int32_t)row0);
                    bulk_load(sSF + stage * C::SFP_BYTES, sf + (int64_t)kb * 4 * 512, C::SFP_BYTES, full + stage);
                    issued |= 1u << stage;
                    issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // copies in flight land within microseconds; each wait stops at 1 ms
                WaitCfg w2 = wc;
                if (w2.limit_ns > 1000000ull) w2.limit_ns = 1000000ull;
                volatile int never = 0;
                for (int s = 0; s < C::STAGES; ++s)
                    if ((issued >> s) & 1u) mbar_wait(full + s, (issued_ph >> s) & 1u, w2, &never);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_mxf4(128, C::BN, false);
            int stage = 0;
            uint32_t ph = 0;
            bool ok = true, any = false;
            int n = 0;
            for (int v = blockIdx.x; v < U && ok; v += gridDim.x, ++n) {
                bool g1;
                int ai, t;
                unit(v, g1, ai, t);
                const int b = n & 1;
                const uint32_t par = (uint32_t)(n >> 1) & 1u;
                // accumulator b has been read (unit n - 2), token tile b is written (unit n)
                if (!mbar_wait(acce + b, par ^ 1u, wc, abort_flag) || !mbar_wait(qfull + b, par, wc, abort_flag))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(b * C::BN);
                const uint32_t qc0 = smem_u32(sQ + b * C::QBUF);
                const int kbn = g1 ? kb1 : kb2;
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!mbar_wait(full + stage, ph, wc, abort_flag) ||
                        !mbar_wait(tready + stage, ph, wc, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfp_t = tmem + (uint32_t)(2 * C::BN + stage * C::SF_COLS);
                    const uint32_t sfq_t = sfp_t + 16;
                    const uint32_t pa = smem_u32(sP + stage * C::P_BYTES);
                    const uint32_t qa = qc0 + kb * C::QC_BYTES;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf4<false>(d_tmem, sdesc_sw128(pa + kk * 32), sdesc_sw128(qa + kk * 32), idesc,
                                        sfp_t + kk * 4, sfq_t + kk * 4, (kb > 0 || kk > 0) ? 1u : 0u);
                    any = true;
                    mma_commit(empty + stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(accf + b);
                mma_commit(qempty + b);
            }
            if (any && *abort_flag) {
                // the tensor-core work already issued finishes before TMEM is freed
                mma_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, wc, &never);
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------ token operand tiles (warps 12-15)
        const int q = threadIdx.x - 384;  // 0..127
        int n = 0;
        for (int v = blockIdx.x; v < U; v += gridDim.x, ++n) {
            bool g1;
            int ai, t;
            unit(v, g1, ai, t);
            const int e = s_act[ai];
            const int ne = s_ne[ai];
            const int qb = n & 1;
            // 1. tile qb is free (the MMAs of unit n - 2 are done) and the unit's
            //    global scale is known (GEMM2: after the expert's GEMM1 units)
            if (q == 0) {
                bool ok = mbar_wait(qempty + qb, ((uint32_t)(n >> 1) & 1u) ^ 1u, wc, abort_flag);
                float sg = 0.0f;
                if (ok) {
                    if (g1) {
                        sg = a.is_static ? st.s13[e] : sg_a;
                    } else {
                        ok = wait_count(a.cnt1 + ai, (uint32_t)n1, wc, abort_flag);
                        const float amax = __uint_as_float(ld_acquire_u32(a.amax_h + ai));
                        sg = a.is_static ? st.s2[e] : __fdiv_rn(amax, 2688.0f);
                        if (ok && t == 0) a.sg_h[e] = sg;
                        s_sgh[ai] = sg;  // for the epilogue (ordered by the tile's barriers)
                    }
                }
                s_misc[3] = (int32_t)__float_as_uint(sg);
                s_misc[4] = ok ? 0 : 1;  // one decision for the group (named barriers follow)
            }
            named_bar_sync(3, 128);
            if (s_misc[4]) break;
            const float sg = __uint_as_float((uint32_t)s_misc[3]);
            const int K = g1 ? H : I;
            const int bpr = K / 16;  // blocks per row
            const int nbb = ne * bpr;
            // the source of block bb (row r = bb / bpr of the unit's tokens, block j):
            // the hidden row of its token, or (GEMM2) the slot's h row, written by
            // other CTAs before the counter the decision above waited for
            auto load_blk = [&](int bb, uint4& x0, uint4& x1) {
                const int r = bb / bpr, j = bb - r * bpr;
                const int slot = s_eslot[ai * kFusedMaxT + r];
                if (g1) {
                    const uint4* src = reinterpret_cast<const uint4*>(a.hidden + (int64_t)(slot / k) * H + j * 16);
                    x0 = __ldg(src);
                    x1 = __ldg(src + 1);
                } else {
                    const uint4* src = reinterpret_cast<const uint4*>(a.h + (int64_t)slot * I + j * 16);
                    x0 = __ldcg(src);
                    x1 = __ldcg(src + 1);
                }
            };
            // the thread's first block is in flight while the divisors are formed
            uint4 xn0 = make_uint4(0u, 0u, 0u, 0u), xn1 = xn0;
            if (q < nbb) load_blk(q, xn0, xn1);
            float2* tab = dtab;  // GEMM1, dynamic scale: the prologue's table
            // one or two tokens (at most one block per thread): each thread takes
            // its block's divisor itself (the table's entry for that byte, with the
            // same refinement) instead of the table and its barrier
            const bool direct = ne <= 2 && nbb <= 128;
            if ((!g1 || a.is_static) && !direct) {
                tab = dtab + (1 + qb) * 128;
                tab[q] = nvfp4_divisor((uint32_t)q, sg, ne > 2);
                named_bar_sync(3, 128);
            }
            const float p_t = __fmul_rn(sg, 6.0f);
            const float inv_p = nvfp4_inv_p(p_t);
            // 2. ne rows x K, NVFP4 with s_g = sg, straight into the MMA's swizzled
            //    tile (row r, K block kb, 16-byte piece c at piece c ^ (r % 8)) and
            //    scale atoms (row r at r * 16)
            uint8_t* qc = sQ + qb * C::QBUF;
            uint8_t* qs = qc + C::MAX_KB * C::QC_BYTES;
            const bool dump = t == 0;  // one unit per expert leaves the codes in the workspace
            for (int bb = q; bb < nbb; bb += 128) {
                const int r = bb / bpr, j = bb - r * bpr;
                const int slot = s_eslot[ai * kFusedMaxT + r];
                const uint4 x0 = xn0, x1 = xn1;
                if (bb + 128 < nbb) load_blk(bb + 128, xn0, xn1);  // the next block in flight
                uint32_t am = absmax8(x1, absmax8(x0, 0u));
                am = max(am & 0xFFFFu, am >> 16);
                const uint32_t sbyte = nvfp4_scale_byte(__uint_as_float(am << 16), p_t, inv_p);
                const float2 dv = (!g1 || a.is_static) && direct ? nvfp4_divisor(sbyte, sg, ne > 2) : tab[sbyte];
                float f[8];
                unpack8(x0, f);
                const uint32_t w0 = nvfp4_word(f, dv);
                unpack8(x1, f);
                const uint32_t w1 = nvfp4_word(f, dv);
                const int kb = j >> 4, jj = j & 15;
                const uint32_t qa = smem_u32(qc + kb * C::QC_BYTES) + (uint32_t)r * 128u +
                                    ((((uint32_t)jj >> 1) ^ ((uint32_t)r & 7u)) << 4) + (((uint32_t)jj & 1u) << 3);
                asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(qa), "r"(w0), "r"(w1) : "memory");
                qs[kb * C::QS_BYTES + (jj >> 2) * 128 + r * 4 + (jj & 3)] = (uint8_t)sbyte;
                if (dump) {
                    uint8_t* dc = g1 ? a.a_codes + (int64_t)slot * (H / 2) : a.h_codes + (int64_t)slot * (I / 2);
                    uint8_t* ds = g1 ? a.a_sbytes + (int64_t)slot * (H / 16) : a.h_sbytes + (int64_t)slot * (I / 16);
                    *reinterpret_cast<uint2*>(dc + j * 8) = make_uint2(w0, w1);
                    ds[j] = (uint8_t)sbyte;
                }
            }
            fence_proxy_async();  // the tile is read by the tensor cores
            named_bar_sync(3, 128);
            if (q == 0) mbar_arrive(qfull + qb);
        }
    } else if (warp >= 8) {
        // --------------------------------------------------- epilogue (warps 8-11)
        const int qd = warp - 8;
        int n = 0;
        for (int v = blockIdx.x; v < U; v += gridDim.x, ++n) {
            bool g1;
            int ai, t;
            unit(v, g1, ai, t);
            const int e = s_act[ai];
            const int ne = s_ne[ai];
            const int b = n & 1;
            if (threadIdx.x == 256) s_misc[5] = mbar_wait(accf + b, (uint32_t)(n >> 1) & 1u, wc, abort_flag) ? 0 : 1;
            named_bar_sync(2, 128);
            if (s_misc[5]) break;  // one decision for the group
            tc_fence_after();
            {
                // the accumulator's first kFusedMaxT columns (the expert's tokens) of this
                // lane quarter, alpha-scaled, into xq[column][lane]: the loops below run
                // over the unit's tokens only (short code, run once per unit)
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(b * C::BN), r);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce + b);
                const float alpha = g1 ? __fmul_rn(a.is_static ? st.s13[e] : sg_a, s_gw13[e])
                                       : __fmul_rn(s_sgh[ai], s_gw2[e]);
                float* xq = sX + qd * kFusedMaxT * 32;
#pragma unroll
                for (int c = 0; c < kFusedMaxT; ++c) xq[c * 32 + lane] = __fmul_rn(alpha, __uint_as_float(r[c]));
            }
            named_bar_sync(2, 128);
            if (g1) {
                // W13 rows interleaved in groups of 32: quarters 0 / 1 hold gate / up
                // of features 64 t + [0, 32), quarters 2 / 3 of 64 t + [32, 64)
                if (qd & 1) {
                    const float* xg = sX + (qd - 1) * kFusedMaxT * 32;
                    const float* xu = sX + qd * kFusedMaxT * 32;
                    const int f = t * 64 + (qd >> 1) * 32 + lane;
                    uint32_t amax_bits = 0;
#pragma unroll 1
                    for (int c = 0; c < ne; ++c) {
                        const __nv_bfloat16 hb = __float2bfloat16_rn(__fmul_rn(silu_f32(xg[c * 32 + lane]), xu[c * 32 + lane]));
                        const uint16_t hbits = *reinterpret_cast<const uint16_t*>(&hb);
                        a.h[(int64_t)s_eslot[ai * kFusedMaxT + c] * I + f] = hbits;
                        amax_bits = max(amax_bits, (uint32_t)(hbits & 0x7FFFu));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        amax_bits = max(amax_bits, __shfl_xor_sync(0xFFFFFFFFu, amax_bits, o));
                    if (lane == 0 && amax_bits) atomicMax(a.amax_h + ai, amax_bits << 16);
                }
                named_bar_sync(2, 128);
                if (threadIdx.x == 256) {
                    fence_acq_rel_gpu();
                    atomicAdd(a.cnt1 + ai, 1u);
                }
            } else {
                const float* xq = sX + qd * kFusedMaxT * 32;
                const int f = t * 128 + qd * 32 + lane;
#pragma unroll 1
                for (int c = 0; c < ne; ++c) a.d[(int64_t)s_eslot[ai * kFusedMaxT + c] * H + f] = xq[c * 32 + lane];
                named_bar_sync(2, 128);
                if (threadIdx.x == 256) {
                    fence_acq_rel_gpu();
                    const uint32_t old = atomicAdd(a.cnt2 + t, 1u);
                    s_misc[2] = old + 1u == (uint32_t)E_act ? 1 : 0;
                }
                named_bar_sync(2, 128);
                if (s_misc[2]) {
                    // the last expert of this output tile: the top-k sum in slot order,
                    // four tokens' loads in flight at a time
                    fence_acq_rel_gpu();
                    const int fo = t * 128 + (threadIdx.x - 256);
                    for (int tok0 = 0; tok0 < T; tok0 += 4) {
                        float dv[4][kFusedMaxTopK];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int j = 0; j < kFusedMaxTopK; ++j)
                                dv[u][j] = (tok0 + u < T && j < k) ? __ldcg(a.d + (int64_t)((tok0 + u) * k + j) * H + fo)
                                                                    : 0.0f;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (tok0 + u >= T) break;
                            float y = 0.0f;
#pragma unroll
                            for (int j = 0; j < kFusedMaxTopK; ++j)
                                if (j < k) y = __fadd_rn(y, __fmul_rn(s_w[(tok0 + u) * k + j], dv[u][j]));
                            const __nv_bfloat16 yb = __float2bfloat16_rn(y);
                            a.out[(int64_t)(tok0 + u) * H + fo] = *reinterpret_cast<const uint16_t*>(&yb);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

static PFN_cuTensorMapEncodeTiled_v12000 fused_encode_fn() {
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

static bool weight_map(CUtensorMap* m, const void* codes, int64_t rows, int64_t k) {
    auto fn = fused_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t es[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool moe_fused_supported(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
    return T >= 1 && T <= kFusedMaxT && k >= 1 && k <= kFusedMaxTopK && E <= kFusedMaxE && H % 256 == 0 &&
           H <= kFusedMaxK && H / 128 <= kFusedMaxOutTiles && I % 256 == 0 && I <= kFusedMaxK;
}

cudaError_t launch_moe_fused(const FusedMoeLaunch& L, const StaticScales& st, cudaStream_t s) {
    using C = FusedCfg;
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    CUtensorMap tm13, tm2;
    if (!weight_map(&tm13, L.w13_codes, L.E * 2 * L.I, L.H) || !weight_map(&tm2, L.w2_codes, L.E * L.H, L.I)) {
        set_error("cuTensorMapEncodeTiled failed for the expert weights");
        return cudaErrorInvalidValue;
    }
    FusedMoeArgs a;
    a.hidden = L.hidden;
    a.logits = L.logits;
    a.T = (int)L.T;
    a.H = (int)L.H;
    a.I = (int)L.I;
    a.E = (int)L.E;
    a.k = (int)L.k;
    a.is_static = L.is_static;
    a.w13_scales = L.w13_scales;
    a.w13_global = L.w13_global;
    a.w2_scales = L.w2_scales;
    a.w2_global = L.w2_global;
    a.out = L.out;
    a.ids = L.ids;
    a.weights = L.weights;
    a.sg_a = L.sg_a;
    a.cnt1 = L.zeroed;
    a.cnt2 = L.zeroed + kFusedMaxSlots;
    a.amax_h = L.zeroed + kFusedMaxSlots + kFusedMaxOutTiles;
    a.h = L.h;
    a.a_codes = L.a_codes;
    a.a_sbytes = L.a_sbytes;
    a.h_codes = L.h_codes;
    a.h_sbytes = L.h_sbytes;
    a.sg_h = L.sg_h;
    a.d = L.d;
    // clear the counters and the amax (one small memset), then the kernel
    if (cudaError_t e = cudaMemsetAsync(L.zeroed, 0, kFusedZeroedBytes, s)) return e;
    const int per_lane = (int)((L.E + 31) / 32);
    const void* fn = per_lane <= 4    ? (const void*)moe_fused_kernel<4>
                     : per_lane <= 8  ? (const void*)moe_fused_kernel<8>
                     : per_lane <= 16 ? (const void*)moe_fused_kernel<16>
                                      : (const void*)moe_fused_kernel<32>;
    static uint64_t done[4] = {0, 0, 0, 0};
    const int which = per_lane <= 4 ? 0 : per_lane <= 8 ? 1 : per_lane <= 16 ? 2 : 3;
    if (cudaError_t e = set_smem_attr_once(fn, C::SMEM, done[which])) return e;
    // units: every active expert's GEMM1 and GEMM2 tiles (at most T k experts)
    const int64_t e_act_max = L.T * L.k < L.E ? L.T * L.k : L.E;
    const int64_t units = e_act_max * (2 * L.I / 128 + L.H / 128);
    int64_t grid = d->sm_count;
    if (units < grid) grid = units;
    WaitCfg wc;
    wc.limit_ns = wait_limit_ns();
    wc.err = d->err_word;
    StaticScales sc = st;
    void* args[] = {(void*)&tm13, (void*)&tm2, (void*)&a, (void*)&sc, (void*)&wc};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: CTAs wait on one another
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace fp4
