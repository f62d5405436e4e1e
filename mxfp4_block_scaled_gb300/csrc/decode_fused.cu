// decode_fused.cu -- the small-M (decode) W4A4 linear in one launch.
//
// out[t][n] = bf16(alpha * sum_k deq(A)[t][k] * deq(W)[n][k]) for t < m <= 8,
// with A = the bf16 activations quantised in this kernel (dynamic or static
// per-tensor scale, the arithmetic of quant_math.cuh, so the codes are those
// fp4_quantize_act gives) and W the prepacked FP4 weights.  The call streams
// W, so the weight tiles start loading right after the set-up barrier and the
// activations' work runs under that stream:
//
//   one CTA per 128-row weight tile, the whole K (no split, no reduction);
//   MMA: swap-AB, M = 128 weight rows, N = 32 activation rows (rows >= m
//   carry zero scales and feed only accumulator columns nobody reads), K = 64
//   per instruction, four per 256-element K block; the ring's depth is chosen
//   per launch from the shared memory the compact copy leaves;
//   warp 4      TMA producer of the weight tiles (128 rows x 128 B, 128-byte
//               swizzle) -- no dependency wait;
//   warp 7      bulk copies of the weight scale atoms into the scale ring;
//   warps 0-3, 6, 8-15  first, after the dependency wait (their loads go out
//               before the set-up barrier): the activations'
//               abs-max, then all m x K activations quantised once into a
//               compact smem copy (codes [m][K/2], scale bytes [m][K/16 or
//               K/32]), the first ring-full of K blocks also straight into
//               their stages' operand tiles (the MMA's swizzled layout) and
//               scale slots (the MMA scale layout), which warp 8 then marks
//               full; warp 6 copies each later K block from the compact copy
//               when its stage comes free;
//   warps 0-3   scale writers (smem -> TMEM, tcgen05.st), as in gemm_kernel;
//   warp 5      TMEM allocation and the MMA issuer;
//   warps 8-11  epilogue: one tcgen05.ld per lane quarter, alpha, bf16.
//
// Every wait is bounded; on expiry the role sets the device error word and
// an abort flag that stops the others.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "quant_math.cuh"

namespace fp4 {

template <bool MX>
struct DecCfg {
    static constexpr int BN = 32;                  // activation rows on the MMA N side
    static constexpr int KB_BYTES = 128;           // 256 FP4 per row per K block
    static constexpr int SF_CHUNKS = MX ? 2 : 4;   // 512-byte scale atoms per 128 rows per K block
    static constexpr int P_BYTES = 128 * KB_BYTES;
    static constexpr int Q_BYTES = BN * KB_BYTES;
    static constexpr int SFP_BYTES = SF_CHUNKS * 512;
    static constexpr int SFQ_BYTES = SF_CHUNKS * 512;
    static constexpr int STAGE_BYTES = P_BYTES + Q_BYTES + SFP_BYTES + SFQ_BYTES;
    static constexpr int SF_COLS = 2 * SF_CHUNKS * 4;  // P and Q scale columns per stage
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    static constexpr int MAX_K = (int)kDecodeFusedMaxK;  // fused path: k <= MAX_K
    static constexpr int DTAB = 128 * 8;                 // NVFP4 divisor entry per scale byte
    static constexpr int FIXED = 1024 + BAR_BYTES + DTAB;  // alignment slack, barriers, divisor table
    // The ring holds as many stages as the shared memory left beside the
    // compact activation copy (m rows of codes and scale bytes) takes, up to
    // MAX_STAGES: the K blocks beyond the ring wait a full copy round trip
    // each time the ring turns, so for K = 4096 (16 K blocks) 8 stages take
    // two turns where 7 take three.
    static constexpr int MAX_STAGES = 12;
    static constexpr int ST_TMEM = (512 - BN) / SF_COLS;
    static constexpr int64_t compact_bytes(int m, int64_t k) {
        return ((int64_t)m * (k / 2 + k / (MX ? 32 : 16)) + 15) / 16 * 16;
    }
    static constexpr int stages(int m, int64_t k) {
        const int64_t by_smem = (SMEM_LIMIT - FIXED - compact_bytes(m, k)) / STAGE_BYTES;
        int64_t st = by_smem < ST_TMEM ? by_smem : ST_TMEM;
        return (int)(st < MAX_STAGES ? st : MAX_STAGES);
    }
    static constexpr int64_t smem_bytes(int m, int64_t k) {
        return FIXED + (int64_t)stages(m, k) * STAGE_BYTES + compact_bytes(m, k);
    }
    static_assert(4 * MAX_STAGES + 4 <= BAR_BYTES / 8 - 4, "barrier area too small");
    static_assert(ST_TMEM >= MAX_STAGES, "TMEM scale columns");
    static_assert(stages(kDecodeFusedMaxM, MAX_K) >= 4, "pipeline too shallow at the largest m and K");
    static_assert(smem_bytes(kDecodeFusedMaxM, MAX_K) <= SMEM_LIMIT, "shared memory budget");
};

struct DecodeArgs {
    const uint16_t* x;     // bf16 activations [m][k]
    int m;                 // 1..8
    int64_t k, n;
    const uint8_t* w_scales;
    const float* w_global;  // NVFP4: one fp32 (device)
    int dynamic;            // NVFP4: 1 = s_g from the activations' amax, 0 = static_scale
    float static_scale;
    float* a_global_out;    // optional: the activation s_g (device), written by CTA 0
    uint16_t* out;          // bf16 [m][n]
    int stages;             // ring depth, DecCfg::stages(m, k)
};

template <bool MX>
__global__ void __launch_bounds__(512, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap tmW, const DecodeArgs a, const WaitCfg wc) {
    using C = DecCfg<MX>;
    extern __shared__ uint8_t smem_raw[];
    const int NS = a.stages;
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* sP = smem;
    uint8_t* sQ = sP + NS * C::P_BYTES;
    uint8_t* sSFP = sQ + NS * C::Q_BYTES;
    uint8_t* sSFQ = sSFP + NS * C::SFP_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sSFQ + NS * C::SFQ_BYTES);
    uint64_t* full = bars;            // weight tile + activation tile + scales in TMEM
    uint64_t* empty = bars + NS;      // the stage's MMAs are complete
    uint64_t* sfull = bars + 2 * NS;  // weight scale atoms landed + activation scales written
    uint64_t* sempty = bars + 3 * NS; // the writers are done with the scale slot
    uint64_t* accf = bars + 4 * NS;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(accf + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
    float* s_sg = reinterpret_cast<float*>(tslot + 2);
    uint32_t* s_red = tslot + 4;  // 16 words
    float2* dtab = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(bars) + C::BAR_BYTES);
    uint8_t* xc = reinterpret_cast<uint8_t*>(dtab) + C::DTAB;         // compact codes [m][k/2]
    const int64_t cb = a.k / 2;                                       // code bytes per row
    const int64_t sbpr = a.k / (MX ? 32 : 16);                        // scale bytes per row
    uint8_t* xs = xc + a.m * cb;                                      // compact scale bytes [m][sbpr]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tile = blockIdx.x;  // 128 weight rows
    const int64_t kbt = (a.k + 255) / 256;
    const int64_t ksfc = kbt * C::SF_CHUNKS;  // scale atoms per 128-row tile

    // The activation threads (warps 0-3, 6, 8-15) issue their loads first, so
    // that the latency runs under the setup (the weight stream starts after
    // it: issued first, its copies would queue these loads behind them, and
    // a TMA issue stalls while the copy engine's queue is full, which would
    // hold up the setup barrier).  A thread takes 8-element chunks
    // i = ta + 416 j, and the first R rounds' chunks stay in registers for the
    // abs-max and the quantisation (all of them for m k <= R x 416 x 8 =
    // 39,936 elements, e.g. 8 rows of 4096).
    constexpr int NT = 416;
    constexpr int R = 12;
    const bool act_warp = warp < 4 || warp == 6 || warp >= 8;
    const int ta = warp < 4 ? warp * 32 + lane : warp == 6 ? 128 + lane : 160 + (warp - 8) * 32 + lane;
    const uint32_t nvec = (uint32_t)((int64_t)a.m * a.k / 8);  // < 2^16 (m <= 8, k <= 8192)
    const uint4* xv = reinterpret_cast<const uint4*>(a.x);
    uint4 v0[R];
    if (act_warp) {
        pdl_wait();
#pragma unroll
        for (int u = 0; u < R; ++u) v0[u] = ta + u * NT < nvec ? __ldg(xv + ta + u * NT) : make_uint4(0u, 0u, 0u, 0u);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full + s, 6);   // weight producer + activation quantiser + 4 scale writers
            mbar_init(empty + s, 1);
            mbar_init(sfull + s, 2);  // weight-scale producer + activation quantiser
            mbar_init(sempty + s, 4);
        }
        mbar_init(accf, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmW);
    }
    // The activation scale slots start zeroed: the scale bytes past K in a last
    // partial K block, and those of rows >= m, are never written.  The operand
    // tiles' rows >= m are left as they are: they only feed accumulator columns
    // >= m, which nothing reads, and E2M1 codes are finite whatever the bits.
    for (int i = threadIdx.x; i < NS * C::SFQ_BYTES / 16; i += 512)
        reinterpret_cast<uint4*>(sSFQ)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async();  // the zeros are visible to the tensor core's reads
    if (warp == 5) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    // the next kernel may be scheduled now (its weight stream overlaps this
    // one's tail); it waits for this grid's completion before reading the output
    pdl_launch_dependents();

    // ------------------------------------------------------------------
    // The activations (the weight producers and the MMA issuer go straight to
    // their loops): abs-max and s_g, then the compact quantised copy.  Lanes
    // 2l, 2l+1 (4l..4l+3) hold the chunks of one NVFP4 (MXFP4) block.
    float sg = a.static_scale;
    if (act_warp) {
        if (!MX && a.dynamic) {
            uint32_t mx = 0;
#pragma unroll
            for (int u = 0; u < R; ++u) mx = absmax8(v0[u], mx);
            for (uint32_t i0 = ta + R * NT; i0 < nvec; i0 += 4 * NT) {  // four loads in flight
                uint4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = i0 + u * NT < nvec ? __ldg(xv + i0 + u * NT) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4; ++u) mx = absmax8(v[u], mx);
            }
            mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            if (lane == 0) s_red[ta >> 5] = mx;
            named_bar_sync(1, NT);
            if (ta == 0) {
                uint32_t v = 0;
                for (int i = 0; i < NT / 32; ++i) v = max(v, s_red[i]);
                *s_sg = __fdiv_rn(__uint_as_float(v << 16), 2688.0f);
            }
            named_bar_sync(1, NT);
            sg = *s_sg;
        }
        if (blockIdx.x == 0 && ta == 0 && a.a_global_out) *a.a_global_out = MX ? 1.0f : sg;
        // NVFP4: the divisor entry of each scale byte (nvfp4_divisor)
        const float p_t = __fmul_rn(sg, 6.0f);
        const float inv_p = nvfp4_inv_p(p_t);
        // (the one-value test and neighbour search of the table make almost every
        // block take the one-multiply path; for a single row the table is on the
        // critical path and the per-element bracket costs less)
        if (!MX && ta < 128) dtab[ta] = nvfp4_divisor((uint32_t)ta, sg, a.m > 1);
        named_bar_sync(1, NT);
        constexpr int LPB = MX ? 4 : 2;  // lanes per block
        const uint32_t cpr = (uint32_t)(a.k / 8);  // chunks per row
        // Four rounds of chunks at a time; the trip counts follow the warp's first
        // chunk, so they are the same for all lanes of the warp (the shuffles
        // below need every lane).
        const uint32_t dr = NT / cpr, dc = NT - dr * cpr;  // a round's step in (row, chunk)
        auto convert4 = [&](const uint4 (&vb)[4], uint32_t jb) {
            const uint32_t j0 = jb + (uint32_t)lane;
            uint32_t r = j0 / cpr, c = j0 - r * cpr;  // row and chunk of round u, stepped below
#pragma unroll
            for (int u2 = 0; u2 < 4; u2 += 2) {
                // Rounds go in pairs whose arithmetic overlaps (its stores come
                // after both); a pair that starts beyond the activations is empty
                // for the whole warp (jb is its first chunk): few rows leave most
                // rounds empty.
                if (jb + (uint32_t)(u2 * NT) >= nvec) break;
                uint32_t w[2], sbyte[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // every lane takes part in the shuffles; nvec and the chunks per row are
                    // multiples of 4 (k % 32 == 0), so a block's lanes are all in or all out
                    const uint4 v = vb[u2 + h];
                    uint32_t am = absmax8(v, 0u);
                    am = max(am & 0xFFFFu, am >> 16);
                    am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
                    if (MX) am = max(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
                    const float amax_b = __uint_as_float(am << 16);
                    if constexpr (!MX) {
                        sbyte[h] = nvfp4_scale_byte(amax_b, p_t, inv_p);
                        float f[8];
                        unpack8(v, f);
                        w[h] = nvfp4_word(f, dtab[sbyte[h]]);
                    } else {
                        float inv;
                        sbyte[h] = mxfp4_scale_byte(amax_b, inv);
                        w[h] = mxfp4_codes8(v, inv);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (j0 + (uint32_t)((u2 + h) * NT) < nvec) {
                        *reinterpret_cast<uint32_t*>(xc + (int64_t)r * cb + c * 4) = w[h];
                        if ((lane & (LPB - 1)) == 0) xs[(int64_t)r * sbpr + c / LPB] = (uint8_t)sbyte[h];
                        // the first NS K blocks (32 chunks each) also go straight into
                        // their stage's operand tile and scale slot, in the layout warp 6
                        // gives the later ones, so the first MMAs do not wait for its copy
                        const uint32_t kbi = c >> 5, cc = c & 31;
                        if (kbi < (uint32_t)NS) {
                            *reinterpret_cast<uint32_t*>(sQ + kbi * (uint32_t)C::Q_BYTES + r * 128u +
                                                         (((cc >> 2) ^ (r & 7u)) << 4) + ((cc & 3u) << 2)) = w[h];
                            const uint32_t jblk = cc / LPB;  // scale block within the K block
                            if ((lane & (LPB - 1)) == 0)
                                sSFQ[kbi * C::SFQ_BYTES + (jblk >> 2) * 512 + r * 16 + (jblk & 3)] = (uint8_t)sbyte[h];
                        }
                    }
                    r += dr;
                    c += dc;
                    if (c >= cpr) {
                        c -= cpr;
                        ++r;
                    }
                }
            }
        };
        const uint32_t jw = (uint32_t)(ta & ~31);
#pragma unroll
        for (int it = 0; it < R / 4; ++it) {  // the rounds held in registers
            const uint32_t jb = jw + (uint32_t)(it * 4 * NT);
            if (jb >= nvec) break;  // warp-uniform
            const uint4 vb[4] = {v0[4 * it], v0[4 * it + 1], v0[4 * it + 2], v0[4 * it + 3]};
            convert4(vb, jb);
        }
        for (uint32_t jb = jw + R * NT; jb < nvec; jb += 4 * NT) {  // the rest, loaded
            const uint32_t j0 = jb + (uint32_t)lane;
            uint4 vb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) vb[u] = j0 + u * NT < nvec ? __ldg(xv + j0 + u * NT) : make_uint4(0u, 0u, 0u, 0u);
            convert4(vb, jb);
        }
        fence_proxy_async();    // the stage tiles written above are read by the tensor core
        named_bar_sync(1, NT);  // the compact copy (and the first NS stages' tiles) are complete
        if (warp == 8 && lane < (kbt < NS ? (int)kbt : NS)) {
            // the activation part of the first turn of the ring is in place: a
            // warp that has nothing else to do until the epilogue says so, lane
            // s for stage s
            mbar_arrive(full + lane);
            mbar_arrive(sfull + lane);
        }
    }

    if (warp < 4) {
        // ---------------------------------------------------- scale writers
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        uint32_t ph = 0;
        int stage = 0;
        for (int64_t kb = 0; kb < kbt; ++kb) {
            if (!mbar_wait(sfull + stage, ph, wc, abort_flag) || !mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag))
                break;
            const uint32_t sfp_t = tmem + lane_base + (uint32_t)(C::BN + stage * C::SF_COLS);
            const uint32_t sfq_t = sfp_t + C::SF_CHUNKS * 4;
            const uint32_t sp = smem_u32(sSFP + stage * C::SFP_BYTES) + lane * 16;
            const uint32_t sq = smem_u32(sSFQ + stage * C::SFQ_BYTES) + lane * 16;
#pragma unroll
            for (int c = 0; c < C::SF_CHUNKS; ++c) {
                tmem_st4(sfp_t + c * 4, lds128(sp + c * 512));
                tmem_st4(sfq_t + c * 4, lds128(sq + c * 512));
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(full + stage);
                mbar_arrive(sempty + stage);
            }
            if (++stage == NS) {
                stage = 0;
                ph ^= 1u;
            }
        }
    } else if (warp == 4 || warp == 7) {
        if (lane == 0) {
            // ------------------------------------------------ weight producers
            // (weights do not depend on the preceding kernel: no dependency wait)
            const bool is_sf = warp == 7;
            uint32_t ph = 0;
            int stage = 0;
            uint32_t issued = 0, issued_ph = 0;
            bool ok = true;
            for (int64_t kb = 0; kb < kbt; ++kb) {
                if (!mbar_wait(is_sf ? sempty + stage : empty + stage, ph ^ 1u, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                if (is_sf) {
                    mbar_arrive_expect_tx(sfull + stage, C::SFP_BYTES);
                    bulk_load(sSFP + stage * C::SFP_BYTES, a.w_scales + (tile * ksfc + kb * C::SF_CHUNKS) * 512,
                              C::SFP_BYTES, sfull + stage);
                } else {
                    mbar_arrive_expect_tx(full + stage, C::P_BYTES);
                    tma_load_2d(&tmW, full + stage, sP + stage * C::P_BYTES, (int32_t)(kb * 128), (int32_t)(tile * 128));
                }
                issued |= 1u << stage;
                issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                if (++stage == NS) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) {
                // copies in flight land within microseconds; a stage's phase may
                // also lack the other roles' arrivals, so each wait stops at 1 ms
                WaitCfg w2 = wc;
                if (w2.limit_ns > 1000000ull) w2.limit_ns = 1000000ull;
                volatile int never = 0;
                for (int s = 0; s < NS; ++s)
                    if ((issued >> s) & 1u)
                        mbar_wait(is_sf ? sfull + s : full + s, (issued_ph >> s) & 1u, w2, &never);
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_mxf4(128, C::BN, MX);
            uint32_t ph = 0;
            int stage = 0;
            bool any = false, ok = true;
            for (int64_t kb = 0; kb < kbt; ++kb) {
                if (!mbar_wait(full + stage, ph, wc, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sfp_t = tmem + (uint32_t)(C::BN + stage * C::SF_COLS);
                const uint32_t sfq_t = sfp_t + C::SF_CHUNKS * 4;
                const uint32_t pa = smem_u32(sP + stage * C::P_BYTES);
                const uint32_t qa = smem_u32(sQ + stage * C::Q_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_sw128(pa + kk * 32);
                    const uint64_t bd = sdesc_sw128(qa + kk * 32);
                    uint32_t sfa, sfb, id;
                    if constexpr (!MX) {
                        sfa = sfp_t + kk * 4;
                        sfb = sfq_t + kk * 4;
                        id = idesc;
                    } else {
                        sfa = sfp_t + (kk >> 1) * 4;
                        sfb = sfq_t + (kk >> 1) * 4;
                        id = idesc_with_sf_id(idesc, (uint32_t)(kk & 1) * 2u);
                    }
                    mma_mxf4<MX>(tmem, ad, bd, id, sfa, sfb, (kb > 0 || kk > 0) ? 1u : 0u);
                }
                any = true;
                mma_commit(empty + stage);
                if (++stage == NS) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            // the accumulator is complete (or, after an abort, the issued MMAs are)
            if (any)
                mma_commit(accf);
            else
                mbar_arrive(accf);
            if (!ok) {
                // the issued MMAs finish before the Tensor Memory is freed
                volatile int never = 0;
                mbar_wait(accf, 0, wc, &never);
            }
        }
    } else {
        // ---------------------------------------------------- warps 6, 8-15
        if (warp == 6) {
            // 3. per K block: the m rows' codes into the stage's operand tile
            //    (row r, 16-byte piece c at piece c ^ (r % 8)), their scale
            //    bytes into the slot (block j at atom j / 4, row r, column j % 4)
            //    from the second turn of the ring on (warp 8 signalled the first)
            constexpr int BPK = MX ? 8 : 16;  // scale blocks per K block
            uint32_t ph = 1;
            int stage = 0;
            for (int64_t kb = NS; kb < kbt; ++kb) {
                // the stage's previous MMAs (and so the writers' reads of the slot) are done
                if (!mbar_wait(empty + stage, ph ^ 1u, wc, abort_flag)) break;
                const uint32_t qbase = smem_u32(sQ + stage * C::Q_BYTES);
                uint8_t* sfq = sSFQ + stage * C::SFQ_BYTES;
                const int64_t byte0 = kb * 128 + lane * 4;  // this lane's 4 code bytes of the K block
                const int64_t col = kb * BPK + lane;         // lanes < BPK: this lane's scale column
                uint32_t w[kDecodeFusedMaxM], sb[kDecodeFusedMaxM];
#pragma unroll
                for (int r = 0; r < kDecodeFusedMaxM; ++r) {  // all rows' reads issued together
                    w[r] = 0u;
                    sb[r] = 0u;
                    if (r < a.m) {
                        if (byte0 < cb) w[r] = *reinterpret_cast<const uint32_t*>(xc + (int64_t)r * cb + byte0);
                        if (lane < BPK && col < sbpr) sb[r] = xs[(int64_t)r * sbpr + col];
                    }
                }
#pragma unroll
                for (int r = 0; r < kDecodeFusedMaxM; ++r) {
                    if (r < a.m) {
                        asm volatile("st.shared.b32 [%0], %1;" ::"r"(qbase + (uint32_t)r * 128u +
                                                                     ((((uint32_t)lane >> 2) ^ ((uint32_t)r & 7u)) << 4) +
                                                                     (((uint32_t)lane & 3u) << 2)),
                                     "r"(w[r])
                                     : "memory");
                        if (lane < BPK) sfq[(lane >> 2) * 512 + r * 16 + (lane & 3)] = (uint8_t)sb[r];
                    }
                }
                fence_proxy_async();  // the operand tile is read by the tensor core
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(full + stage);
                    mbar_arrive(sfull + stage);
                }
                if (++stage == NS) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        } else if (warp < 12) {
            // 3. epilogue: lane quarter warp % 4, all 32 columns (activation rows)
            const int qd = warp & 3;
            if (mbar_wait(accf, 0, wc, abort_flag)) {
                tc_fence_after();
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(qd * 32) << 16), r);
                tmem_ld_wait();
                const float alpha = MX ? 1.0f : __fmul_rn(a.w_global[0], sg);
                const int64_t wrow = tile * 128 + qd * 32 + lane;
                if (wrow < a.n) {
#pragma unroll
                    for (int t = 0; t < kDecodeFusedMaxM; ++t) {  // fixed indices keep r in registers
                        if (t < a.m) {
                            __nv_bfloat16 h = __float2bfloat16_rn(__fmul_rn(alpha, __uint_as_float(r[t])));
                            a.out[(int64_t)t * a.n + wrow] = *reinterpret_cast<uint16_t*>(&h);
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

static PFN_cuTensorMapEncodeTiled_v12000 dec_encode_fn() {
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
static cudaError_t launch_dec(const uint8_t* w_codes, const DecodeArgs& a, bool pdl, cudaStream_t s) {
    using C = DecCfg<MX>;
    auto kern = decode_fused_kernel<MX>;
    static uint64_t attr_done = 0;  // devices on which this instantiation is opted in
    if (cudaError_t e = set_smem_attr_once((const void*)kern, C::SMEM_LIMIT, attr_done)) return e;
    auto fn = dec_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap tm;
    cuuint64_t dims[2] = {(cuuint64_t)(a.k / 2), (cuuint64_t)a.n};
    cuuint64_t strides[1] = {(cuuint64_t)(a.k / 2)};
    cuuint32_t box[2] = {128u, 128u};
    cuuint32_t es[2] = {1u, 1u};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(w_codes), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed for the weights (%lld x %lld)", (long long)a.n, (long long)a.k);
        return cudaErrorInvalidValue;
    }
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    WaitCfg wc;
    wc.limit_ns = wait_limit_ns();
    wc.err = d->err_word;
    DecodeArgs aa = a;
    aa.stages = C::stages(a.m, a.k);
    void* args[] = {(void*)&tm, (void*)&aa, (void*)&wc};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.n + 127) / 128));
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = (size_t)C::smem_bytes(a.m, a.k);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, (const void*)kern, args);
}

cudaError_t launch_decode_fused(int fmt, const uint16_t* x, int m, int64_t n, int64_t k, const uint8_t* w_codes,
                                const uint8_t* w_scales, const float* w_global, int dynamic, float static_scale,
                                float* a_global_out, uint16_t* out, bool pdl, cudaStream_t s) {
    DecodeArgs a;
    a.x = x;
    a.m = m;
    a.k = k;
    a.n = n;
    a.w_scales = w_scales;
    a.w_global = w_global;
    a.dynamic = dynamic;
    a.static_scale = static_scale;
    a.a_global_out = a_global_out;
    a.out = out;
    return fmt == FP4_MXFP4 ? launch_dec<true>(w_codes, a, pdl, s) : launch_dec<false>(w_codes, a, pdl, s);
}

}  // namespace fp4
