// moe.cu -- NVFP4 fused-MoE layer: routing, permutation, grouped expert GEMMs
// with the SwiGLU and combine epilogues, per-expert requantisation.
//
// The stages follow "vLLM on DGX Spark: technical report", section 7.1 (router
// -> quantise/dispatch -> permute, experts, unpermute -> combine) and the
// expert computation of section 4.3 (two GEMMs, SwiGLU, top-k weighted
// reduction).  Launch chain on one stream, no host synchronisation:
//   1 route     top-k per token (a warp per token, 32 tokens per CTA),
//               renormalised weights, expert bitmap; zeroes the h amax
//   2 scan      (one CTA) expert counts, padded offsets (128-row tiles per
//               expert), tile -> expert map; then (a thread per assignment)
//               the row -> (token, slot) and slot -> row maps
//   3 amax      hidden amax partials (dynamic scale)
//   4 dispatch  dynamic scale: each token row quantised once into the rows
//               of its k slots (expert-sorted, padded), padding rows' scale
//               bytes zeroed; static (per-expert) scales: the rows straight
//               into that order under their expert's scale
//   5 GEMM1     grouped tcgen05 GEMM against the interleaved W13, epilogue
//               h = bf16(SiLU(gate) * up) and the per-expert amax of h
//   6 requant   h -> NVFP4 with s_gH[e] = amax_e / 2688
//   7 GEMM2     grouped tcgen05 GEMM against W2, epilogue D[slot] =
//               alpha2 * acc (fp32, one row per routing slot)
//   8 combine   y[t] = bf16(sum over j in slot order of w[t][j] D[t k + j])
// A few tokens (T <= 64) take a one-CTA preparation (route, counts, tables)
// and the swapped grouped GEMMs instead of steps 1-4; at most 16 tokens go to
// the one-launch kernel of moe_fused.cu by default.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "moe_common.cuh"
#include "quant_math.cuh"

namespace fp4 {


// ---------------------------------------------------------------- layout

enum MoeSlot : int {
    MS_IDS = 0,
    MS_WEIGHTS,
    MS_OFFSETS,
    MS_PADDED,
    MS_ROW_SRC,
    MS_A_CODES,
    MS_A_SCALES,
    MS_SG_A,
    MS_H,
    MS_AMAX_H,
    MS_SG_H,
    MS_H_CODES,
    MS_H_SCALES,
    MS_Y,
    MS_PUBLIC_END,  // entry 14 of the public layout is R (the padded row capacity)
    // internal
    MS_BITMAP = MS_PUBLIC_END,
    MS_WPREFIX,
    MS_TILE_EXPERT,
    MS_NPTILES,
    MS_ROW_VALID_END,
    MS_ROW_TOK,
    MS_PARTIALS,
    MS_STATIC13,
    MS_STATIC2,
    MS_SLOT_ROW,    // the expert-sorted row of each slot
    // the one-launch MoE (moe_fused.cu), sized only when its shapes apply
    MS_F_ZERO,      // counters and h amax, cleared per call
    MS_F_H,         // bf16 [T k][I], slot order
    MS_F_HCODES,    // [T k][I/2]
    MS_F_HSB,       // [T k][I/16] scale bytes, row-major
    MS_F_SGH,       // fp32 [E]
    MS_F_D,         // fp32 [T k][H]
    MS_F_ACODES,    // [T k][H/2]
    MS_F_ASB,       // [T k][H/16]
    MS_COUNT
};

struct MoeLayout {
    int64_t off[MS_COUNT];
    int64_t total;
    int64_t R;  // padded row capacity (multiple of 128)
    int64_t W;  // bitmap words per expert
};

static int64_t a256(int64_t x) { return (x + 255) & ~(int64_t)255; }

static MoeLayout moe_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
    MoeLayout L;
    const int64_t slots = T * k;
    const int64_t active = slots < E ? slots : E;
    L.R = round_up(slots + active * 127, 128);
    if (L.R < 128) L.R = 128;
    L.W = (T + 31) / 32;
    int64_t sz[MS_COUNT];
    sz[MS_IDS] = slots * 4;
    sz[MS_WEIGHTS] = slots * 4;
    sz[MS_OFFSETS] = (E + 1) * 4;
    sz[MS_PADDED] = (E + 1) * 4;
    sz[MS_ROW_SRC] = L.R * 4;
    sz[MS_A_CODES] = L.R * H / 2;
    sz[MS_A_SCALES] = L.R * sf_cols_padded(H, 16);
    sz[MS_SG_A] = E * 4;
    sz[MS_H] = L.R * I * 2;
    sz[MS_AMAX_H] = E * 4;
    sz[MS_SG_H] = E * 4;
    sz[MS_H_CODES] = L.R * I / 2;
    sz[MS_H_SCALES] = L.R * sf_cols_padded(I, 16);
    sz[MS_Y] = L.R * H * 4;  // fp32 expert outputs, one row per expert-sorted padded row
    sz[MS_BITMAP] = E * L.W * 4;
    sz[MS_WPREFIX] = E * L.W * 4;
    sz[MS_TILE_EXPERT] = (L.R / 128) * 4;
    sz[MS_NPTILES] = 16;  // [0] token tiles, [1] the most 32-row sub-tiles of a tile
    sz[MS_ROW_VALID_END] = (L.R / 128) * 4;
    sz[MS_ROW_TOK] = L.R * 4;
    sz[MS_PARTIALS] = 4096;
    sz[MS_STATIC13] = E * 4;
    sz[MS_STATIC2] = E * 4;
    sz[MS_SLOT_ROW] = slots * 4;
    const bool fused = moe_fused_supported(T, H, I, E, k);
    sz[MS_F_ZERO] = fused ? kFusedZeroedBytes : 0;
    sz[MS_F_H] = fused ? slots * I * 2 : 0;
    sz[MS_F_HCODES] = fused ? slots * I / 2 : 0;
    sz[MS_F_HSB] = fused ? slots * I / 16 : 0;
    sz[MS_F_SGH] = fused ? E * 4 : 0;
    sz[MS_F_D] = fused ? slots * H * 4 : 0;
    sz[MS_F_ACODES] = fused ? slots * H / 2 : 0;
    sz[MS_F_ASB] = fused ? slots * H / 16 : 0;
    int64_t o = 0;
    for (int i = 0; i < MS_COUNT; ++i) {
        L.off[i] = o;
        o += a256(sz[i] > 0 ? sz[i] : 16);
    }
    L.total = o;
    return L;
}

// ------------------------------------------------------------ kernels

struct RouteArgs {
    const float* logits;
    int64_t T;
    int E, k;
    int32_t* ids;
    float* weights;
    uint32_t* bitmap;  // [E][W]
    int64_t W;
    float* y;          // zeroed: [T*H] fp32
    int64_t y_elems;
    float* amax_h;     // zeroed: [E]
    int route_blocks;
    int has_static;
    float* static13_out;
    float* static2_out;
    int zero_outputs;  // 0: route only (staged runs zero in their own stage)
};

// Route with a warp per token: 32 tokens per CTA of 1024 threads, so the CTA
// owns exactly one 32-token bitmap word per expert (built in smem).  A token's
// top-k takes k rounds of a warp arg-max (topk_token), short enough that a
// handful of tokens costs about what one does.
template <int PER_LANE>
__global__ void __launch_bounds__(1024) moe_route_kernel(const RouteArgs a, const StaticScales st) {
    extern __shared__ uint32_t sbm[];  // [E] bitmap words of this block's 32 tokens
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0) {
        if (a.zero_outputs)
            for (int e = threadIdx.x; e < a.E; e += 1024) a.amax_h[e] = 0.0f;
        if (a.has_static)
            for (int e = threadIdx.x; e < a.E; e += 1024) {
                a.static13_out[e] = st.s13[e];
                a.static2_out[e] = st.s2[e];
            }
    }
    if ((int)blockIdx.x < a.route_blocks) {
        for (int i = threadIdx.x; i < a.E; i += 1024) sbm[i] = 0u;
        __syncthreads();
        const int64_t t = (int64_t)blockIdx.x * 32 + warp;
        if (t < a.T) {
            int e;
            float w;
            topk_token<PER_LANE>(a.logits + t * a.E, a.E, a.k, lane, e, w);
            if (lane < a.k) {
                a.ids[t * a.k + lane] = e;
                a.weights[t * a.k + lane] = w;
                atomicOr(&sbm[e], 1u << warp);
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < a.E; e += 1024) a.bitmap[e * a.W + blockIdx.x] = sbm[e];
    } else if (a.zero_outputs) {
        const int64_t nb = (int64_t)gridDim.x - a.route_blocks;
        float4* y4 = reinterpret_cast<float4*>(a.y);
        const int64_t n4 = a.y_elems / 4;
        for (int64_t i = ((int64_t)blockIdx.x - a.route_blocks) * 1024 + threadIdx.x; i < n4; i += nb * 1024)
            y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

struct ScanArgs {
    const uint32_t* bitmap;  // [E][W]
    int32_t* wprefix;        // [E][W]
    const int32_t* ids;      // [T*k]
    int64_t T, W;
    int E, k;
    int32_t* offsets;        // [E+1]
    int32_t* padded;         // [E+1]
    int32_t* n_ptiles;
    int32_t* tile_expert;    // [R/128]
    int32_t* row_valid_end;  // [R/128]
    int32_t* row_src;        // [R]
    int32_t* row_tok;        // [R]
    int32_t* slot_row;       // [T*k] the row of each routing slot
};

// Exclusive scan of v over the 1024 threads of the block (v = 0 past the data);
// *total receives the sum.
__device__ __forceinline__ int32_t block_exclusive_scan_1024(int32_t v, int32_t* warp_sums, int32_t* total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int32_t ws = warp_sums[lane];
        int32_t wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_sums[lane] = wi - ws;  // exclusive prefix of the warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int32_t r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

// One CTA: counts and word-level prefix counts per expert from the bitmap,
// exclusive scans over experts (plain and padded to 128 rows), the tile map.
// The rows of the assignments come from moe_assign_kernel.
__global__ void __launch_bounds__(1024) moe_scan_kernel(const ScanArgs a) {
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t pad[kMaxExperts + 1];
    __shared__ int32_t wsum[32];
    __shared__ int32_t tot[2];
    __shared__ int32_t cmax;  // the largest expert count
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) cmax = 0;  // dependents wait for this grid's completion
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a warp takes experts warp, warp + 32, ...; their 128-word chunks (four
    // consecutive words a lane) are walked in order with four chunks' loads in
    // flight (a chunk's word prefix needs only the running total of its expert)
    {
        const int nch = (int)((a.W + 127) / 128);
        const int ne = warp < a.E ? (a.E - warp + 31) / 32 : 0;
        const int nit = ne * nch;
        int32_t base = 0;
        for (int it0 = 0; it0 < nit; it0 += 4) {
            uint32_t wv[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int it = it0 + u;
                const int e = warp + 32 * (it / nch), ch = it % nch;
                const int64_t w0 = (int64_t)ch * 128 + lane * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    wv[u][i] = it < nit && w0 + i < a.W ? a.bitmap[(int64_t)e * a.W + w0 + i] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int it = it0 + u;
                if (it >= nit) break;  // warp-uniform
                const int e = warp + 32 * (it / nch), ch = it % nch;
                if (ch == 0) base = 0;
                const int64_t w0 = (int64_t)ch * 128 + lane * 4;
                int32_t c[4], lsum = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    c[i] = __popc(wv[u][i]);
                    lsum += c[i];
                }
                int32_t incl = lsum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += n;
                }
                int32_t pre = base + incl - lsum;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (w0 + i < a.W) a.wprefix[(int64_t)e * a.W + w0 + i] = pre;
                    pre += c[i];
                }
                base += __shfl_sync(0xFFFFFFFFu, incl, 31);
                if (ch == nch - 1 && lane == 0) cnt[e] = base;
            }
        }
    }
    __syncthreads();
    {
        const int e = threadIdx.x;  // E <= 1024 = blockDim
        const int32_t c = e < a.E ? cnt[e] : 0;
        if (c > 0) atomicMax(&cmax, c);
        const int32_t o = block_exclusive_scan_1024(c, wsum, &tot[0]);
        const int32_t p = block_exclusive_scan_1024((c + 127) / 128 * 128, wsum, &tot[1]);
        if (e < a.E) {
            a.offsets[e] = o;
            a.padded[e] = p;
            pad[e] = p;
        }
        if (e == 0) {
            a.offsets[a.E] = tot[0];
            a.padded[a.E] = tot[1];
            pad[a.E] = tot[1];
            *a.n_ptiles = tot[1] / 128;
        }
    }
    __syncthreads();
    // the most 32-row sub-tiles any 128-row token tile holds (the swapped
    // grouped GEMMs schedule no sub-tile beyond it)
    if (threadIdx.x == 0) a.n_ptiles[1] = min(4, (cmax + 31) / 32);
    for (int e = warp; e < a.E; e += 32) {
        const int32_t t0 = pad[e] / 128, t1 = pad[e + 1] / 128;
        for (int32_t t = t0 + lane; t < t1; t += 32) {
            a.tile_expert[t] = e;
            a.row_valid_end[t] = pad[e] + cnt[e];
        }
        for (int32_t r = pad[e] + cnt[e] + lane; r < pad[e + 1]; r += 32) {
            a.row_src[r] = -1;
            a.row_tok[r] = -1;
        }
    }
}

// A thread per assignment (token t, slot s = t * k + j): its row is
// padded[e] + (tokens before t routed to e), from the bitmap and its prefix.
__global__ void __launch_bounds__(256) moe_assign_kernel(const ScanArgs a) {
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    const int64_t slots = a.T * a.k;
    for (int64_t s = (int64_t)blockIdx.x * 256 + threadIdx.x; s < slots; s += (int64_t)gridDim.x * 256) {
        const int64_t t = s / a.k;
        const int e = a.ids[s];
        const int64_t w = t >> 5;
        const uint32_t below = a.bitmap[e * a.W + w] & ((1u << (t & 31)) - 1u);
        const int64_t row = a.padded[e] + a.wprefix[e * a.W + w] + __popc(below);
        a.row_src[row] = (int32_t)s;
        a.row_tok[row] = (int32_t)t;
        a.slot_row[s] = (int32_t)row;
    }
}

// ------------------------------------------------ small-T preparation

// For T <= kPrepMaxTokens the route, the expert counts and scans, the row
// tables and the hidden abs-max run in one CTA of 1024 threads (the other
// CTAs of the launch zero y): at these sizes each is a few microseconds of
// latency.  A 64-bit token mask per expert gives a slot's rank among its
// expert's tokens directly (rows stay in token order).  The quantisation and
// dispatch follow in the same CTA for T <= kPrepInlineTokens (one launch
// replaces six), else in moe_dispatch_kernel across the GPU (the one CTA's
// serial memory round trips would cost more than the launch).  Each token's
// row is quantised once (dynamic scale) and stored to the rows of its k
// slots; with static per-expert scales every slot's row is quantised under
// its expert's scale.  The scale bytes of padding rows are not written: only
// the swapped grouped GEMMs follow this path, and they discard every padding
// column.
static constexpr int kPrepMaxTokens = 64;
static constexpr int kPrepInlineTokens = 16;

struct PrepArgs {
    const float* logits;    // [T][E]
    const uint16_t* hidden; // [T][H] bf16
    int64_t T, H;
    int E, k;
    int32_t* ids;
    float* weights;
    int32_t* offsets;       // [E + 1]
    int32_t* padded;        // [E + 1]
    int32_t* n_ptiles;      // [0] token tiles, [1] most 32-row sub-tiles of a tile
    int32_t* tile_expert;
    int32_t* row_valid_end;
    int32_t* row_src;
    int32_t* row_tok;
    int32_t* slot_row;      // [T*k] expert-sorted row of each slot
    uint8_t* codes;         // expert-sorted rows [R][H/2]
    uint8_t* scales;        // their scale bytes, MMA layout
    float* sg_out;          // dynamic: s_gA
    int has_static;
    int dispatch_inline;    // quantise and dispatch in the preparing CTA
    float* static13_out;
    float* static2_out;
    float* amax_h;          // zeroed [E]
    float* y;               // zeroed [T*H] fp32 by CTAs 1..
    int64_t y_elems;
    float* amax_part;       // [n_amax_ctas] abs-max of a slice of the hidden rows (CTAs 1..)
    int n_amax_ctas;        // dynamic scale, dispatch in moe_dispatch_kernel: CTAs 1.. take the abs-max
    int mark_pad_rows;      // moe_dispatch_kernel: row_src / row_tok = -1 on the tiles' padding rows
    int zero_pad_scales;    // moe_dispatch_kernel: zero scale bytes on the tiles' padding rows
};

// One 16-element block (token t, block column b) of the hidden rows:
// quantised under s_g (divisor entry e, scale-byte divisor p / inv_p) and
// stored to the expert-sorted rows `rows[0..n)`.
__device__ __forceinline__ void prep_block(const PrepArgs& a, int t, int b, int kblocks, int nbp, float p,
                                           float inv_p, float sg, const float2* dtab, const int32_t* rows, int n) {
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (b < kblocks) {
        const uint4* px = reinterpret_cast<const uint4*>(a.hidden + (int64_t)t * a.H + (int64_t)b * 16);
        v0 = __ldg(px);
        v1 = __ldg(px + 1);
    }
    const uint32_t am = absmax8(v1, absmax8(v0, 0u));
    const uint32_t sbyte = nvfp4_scale_byte(__uint_as_float(max(am & 0xFFFFu, am >> 16) << 16), p, inv_p);
    const float2 e = dtab ? dtab[sbyte] : nvfp4_divisor(sbyte, sg, false);
    float f[8];
    unpack8(v0, f);
    const uint32_t w0 = nvfp4_word(f, e);
    unpack8(v1, f);
    const uint32_t w1 = nvfp4_word(f, e);
    // the rows are read eight at a time before the stores (`rows` is global or
    // shared memory; read one by one between stores, no read could move above
    // the store before it, so each read's latency was paid in turn)
    for (int j0 = 0; j0 < n; j0 += 8) {
        int64_t rr[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rr[u] = j0 + u < n ? (int64_t)rows[j0 + u] : -1;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (rr[u] < 0) break;
            if (b < kblocks)
                *reinterpret_cast<uint2*>(a.codes + rr[u] * (a.H / 2) + (int64_t)b * 8) = make_uint2(w0, w1);
            a.scales[sf_offset(rr[u], b, nbp)] = (uint8_t)sbyte;
        }
    }
}

template <int PER_LANE>
__global__ void __launch_bounds__(1024) moe_prep_small_kernel(const PrepArgs a, const StaticScales st) {
    __shared__ uint64_t tokmask[kMaxExperts];
    __shared__ int32_t padv[kMaxExperts + 1];
    __shared__ int32_t s_ids[kPrepMaxTokens * kMaxTopK];
    __shared__ int32_t s_row[kPrepMaxTokens * kMaxTopK];
    __shared__ int32_t wsum[32];
    __shared__ int32_t tot[2];
    __shared__ int32_t cmax;
    __shared__ uint32_t red[32];
    __shared__ float sh_sg;
    __shared__ float2 dtab[128];
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    if (blockIdx.x > 0) {
        if (a.n_amax_ctas > 0) {
            // the abs-max of one slice of the hidden rows (the dispatch reduces the slices)
            const int64_t nv = a.T * a.H / 8;
            const int64_t per = (nv + a.n_amax_ctas - 1) / a.n_amax_ctas;
            const int64_t b0 = ((int64_t)blockIdx.x - 1) * per;
            const int64_t b1 = b0 + per < nv ? b0 + per : nv;
            const uint4* xv = reinterpret_cast<const uint4*>(a.hidden);
            uint32_t m = 0;
            for (int64_t i = b0 + threadIdx.x; i < b1; i += 2 * 1024) {
                const uint4 v0 = __ldg(xv + i);
                const uint4 v1 = i + 1024 < b1 ? __ldg(xv + i + 1024) : make_uint4(0u, 0u, 0u, 0u);
                m = absmax8(v1, absmax8(v0, m));
            }
            m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
            if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
            __syncthreads();
            if (threadIdx.x < 32) {
                uint32_t v = red[threadIdx.x];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
                if (threadIdx.x == 0) a.amax_part[blockIdx.x - 1] = __uint_as_float(v << 16);
            }
        }
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, k = a.k;
    const int T = (int)a.T;
    // the logits of a warp's tokens are loaded first (when they fit the
    // registers), so their latency runs under the table set-up below
    constexpr int RT = kPrepMaxTokens / 32;     // tokens per warp at most
    constexpr bool PRE = PER_LANE <= 8;         // all of them loaded first
    float lg[PRE ? RT : 1][PER_LANE];
    if constexpr (PRE) {
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            const int t = warp + 32 * i;
#pragma unroll
            for (int q = 0; q < PER_LANE; ++q) {
                const int e = q * 32 + lane;
                lg[i][q] = t < T && e < E ? __ldg(a.logits + (int64_t)t * E + e) : -INFINITY;
            }
        }
    }
    for (int e = tid; e < E; e += 1024) {
        tokmask[e] = 0ull;
        a.amax_h[e] = 0.0f;
        if (a.has_static) {
            a.static13_out[e] = st.s13[e];
            a.static2_out[e] = st.s2[e];
        }
    }
    if (tid == 0) cmax = 0;
    __syncthreads();

    // 1. route: a warp per token
    {
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            const int t = warp + 32 * i;
            if (t >= T) break;
            int e;
            float w;
            if constexpr (PRE)
                topk_regs<PER_LANE>(lg[i], E, k, lane, e, w);
            else
                topk_token<PER_LANE>(a.logits + (int64_t)t * E, E, k, lane, e, w);
            if (lane < k) {
                a.ids[t * k + lane] = e;
                a.weights[t * k + lane] = w;
                s_ids[t * k + lane] = e;
                atomicOr(reinterpret_cast<unsigned long long*>(&tokmask[e]), 1ull << t);
            }
        }
    }
    __syncthreads();

    // 2. counts, offsets and 128-row padded offsets (thread e)
    {
        const int e = tid;
        const int32_t c = e < E ? __popcll(tokmask[e]) : 0;
        if (c > 0) atomicMax(&cmax, c);
        const int32_t o = block_exclusive_scan_1024(c, wsum, &tot[0]);
        const int32_t p = block_exclusive_scan_1024((c + 127) / 128 * 128, wsum, &tot[1]);
        if (e < E) {
            a.offsets[e] = o;
            a.padded[e] = p;
            padv[e] = p;
        }
        if (e == 0) {
            a.offsets[E] = tot[0];
            a.padded[E] = tot[1];
            padv[E] = tot[1];
            a.n_ptiles[0] = tot[1] / 128;
        }
    }
    __syncthreads();
    if (tid == 0) a.n_ptiles[1] = min(4, (cmax + 31) / 32);

    // 3. row tables: tiles, padding rows (here only when the dispatch is
    // inline: moe_dispatch_kernel marks them across the GPU), and each slot's
    // row (token order)
    for (int e = warp; e < E; e += 32) {
        const int32_t c = __popcll(tokmask[e]);
        const int32_t t0 = padv[e] / 128, t1 = padv[e + 1] / 128;
        for (int32_t t = t0 + lane; t < t1; t += 32) {
            a.tile_expert[t] = e;
            a.row_valid_end[t] = padv[e] + c;
        }
        if (a.dispatch_inline)
            for (int32_t r = padv[e] + c + lane; r < padv[e + 1]; r += 32) {
                a.row_src[r] = -1;
                a.row_tok[r] = -1;
            }
    }
    for (int s = tid; s < T * k; s += 1024) {
        const int t = s / k, e = s_ids[s];
        const int32_t row = padv[e] + __popcll(tokmask[e] & ((1ull << t) - 1ull));
        a.row_src[row] = s;
        a.row_tok[row] = t;
        s_row[s] = row;
        a.slot_row[s] = row;
    }

    // 4. dynamic: s_gA from the abs-max of the T hidden rows (unless CTAs 1..
    // take it in slices)
    const int64_t H = a.H;
    if (!a.has_static && a.n_amax_ctas == 0) {
        const uint4* xv = reinterpret_cast<const uint4*>(a.hidden);
        uint32_t m = 0;
        const int64_t nv = (int64_t)T * H / 8;
        for (int64_t i = tid; i < nv; i += 4 * 1024) {  // four loads in flight
            uint4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = i + q * 1024 < nv ? __ldg(xv + i + q * 1024) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < 4; ++q) m = absmax8(v[q], m);
        }
        m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) red[warp] = m;
        __syncthreads();
        if (tid == 0) {
            uint32_t v = 0;
            for (int i = 0; i < 32; ++i) v = max(v, red[i]);
            sh_sg = __fdiv_rn(__uint_as_float(v << 16), 2688.0f);
            a.sg_out[0] = sh_sg;
        }
        __syncthreads();
        if (a.dispatch_inline && tid < 128) dtab[tid] = nvfp4_divisor((uint32_t)tid, sh_sg, false);
    }
    if (!a.dispatch_inline) return;
    __syncthreads();

    // 5. quantise and dispatch
    const int nbp = (int)sf_cols_padded(H, 16);  // scale columns per row (padding included)
    const int kblocks = (int)(H / 16);
    if (!a.has_static) {
        const float p = __fmul_rn(sh_sg, 6.0f);
        const float inv_p = nvfp4_inv_p(p);
        for (int item = tid; item < T * nbp; item += 1024) {
            const int t = item / nbp, b = item - t * nbp;
            prep_block(a, t, b, kblocks, nbp, p, inv_p, sh_sg, dtab, s_row + t * k, k);
        }
    } else {
        for (int item = tid; item < T * k * nbp; item += 1024) {
            const int s = item / nbp, b = item - s * nbp;
            const float sg = st.s13[s_ids[s]];
            const float p = __fmul_rn(sg, 6.0f);
            prep_block(a, s / k, b, kblocks, nbp, p, nvfp4_inv_p(p), sg, nullptr, s_row + s, 1);
        }
    }
}

// The quantisation and dispatch of the small-T preparation across the GPU
// (T > kPrepInlineTokens): a thread per (token, block column), or per (slot,
// block column) with static per-expert scales; the slots' rows come from
// the preparing kernel.
__global__ void __launch_bounds__(256) moe_dispatch_kernel(const PrepArgs a, const StaticScales st) {
    __shared__ float2 dtab[128];
    __shared__ float sh_sg;
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    const int64_t H = a.H;
    const int nbp = (int)sf_cols_padded(H, 16);
    const int kblocks = (int)(H / 16);
    const int T = (int)a.T, k = a.k;
    // padding rows of the expert tiles (rows past each tile's real rows)
    if (a.mark_pad_rows || a.zero_pad_scales) {
        const int64_t n = (int64_t)a.n_ptiles[0] * 128;
        for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256)
            if (i >= a.row_valid_end[i >> 7]) {
                if (a.mark_pad_rows) {
                    a.row_src[i] = -1;
                    a.row_tok[i] = -1;
                }
                if (a.zero_pad_scales)
                    for (int c = 0; c < nbp; c += 4)
                        *reinterpret_cast<uint32_t*>(a.scales + sf_offset(i, c, nbp)) = 0u;
            }
    }
    if (!a.has_static) {
        // s_gA = max over the slices' abs-maxima / 2688
        uint32_t m = 0;
        for (int i = threadIdx.x; i < a.n_amax_ctas; i += 256) m = max(m, __float_as_uint(a.amax_part[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        __shared__ uint32_t red[8];
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < 8; ++w) m = max(m, red[w]);
            sh_sg = a.n_amax_ctas > 0 ? __fdiv_rn(__uint_as_float(m), 2688.0f) : a.sg_out[0];
            if (blockIdx.x == 0 && a.n_amax_ctas > 0) a.sg_out[0] = sh_sg;
        }
        __syncthreads();
        const float sg = sh_sg;
        if (threadIdx.x < 128) dtab[threadIdx.x] = nvfp4_divisor(threadIdx.x, sg, false);
        __syncthreads();
        const float p = __fmul_rn(sg, 6.0f);
        const float inv_p = nvfp4_inv_p(p);
        for (int item = blockIdx.x * 256 + threadIdx.x; item < T * nbp; item += gridDim.x * 256) {
            const int t = item / nbp, b = item - t * nbp;
            prep_block(a, t, b, kblocks, nbp, p, inv_p, sg, dtab, a.slot_row + t * k, k);
        }
    } else {
        for (int item = blockIdx.x * 256 + threadIdx.x; item < T * k * nbp; item += gridDim.x * 256) {
            const int s = item / nbp, b = item - s * nbp;
            const float sg = st.s13[a.ids[s]];
            const float p = __fmul_rn(sg, 6.0f);
            prep_block(a, s / k, b, kblocks, nbp, p, nvfp4_inv_p(p), sg, nullptr, a.slot_row + s, 1);
        }
    }
}

// out[t][f] = bf16( sum_{j < k} w[t][j] * d[row of slot t k + j][f] ), the
// top-k terms added in slot order in fp32 (a thread per 4 consecutive
// features; d holds one fp32 row per expert-sorted padded row), so the output
// is the same bits on every run.
__global__ void __launch_bounds__(256) moe_combine_kernel(const float4* __restrict__ d,
                                                          const float* __restrict__ w,
                                                          const int32_t* __restrict__ slot_row, int64_t T, int k,
                                                          int64_t h4, uint2* __restrict__ out) {
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    const int64_t n = T * h4;
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
        const int64_t t = i / h4, f4 = i - t * h4;
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float wj = w[t * k + j];
            const float4 v = d[(int64_t)slot_row[t * k + j] * h4 + f4];
            y.x = __fadd_rn(y.x, __fmul_rn(wj, v.x));
            y.y = __fadd_rn(y.y, __fmul_rn(wj, v.y));
            y.z = __fadd_rn(y.z, __fmul_rn(wj, v.z));
            y.w = __fadd_rn(y.w, __fmul_rn(wj, v.w));
        }
        __nv_bfloat162 a = __floats2bfloat162_rn(y.x, y.y), b = __floats2bfloat162_rn(y.z, y.w);
        out[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
}

// zero n floats (staged runs)
__global__ void __launch_bounds__(256) zero_kernel(float4* __restrict__ p, int64_t n4) {
    pdl_wait();
    pdl_launch_dependents();  // dependents wait for this grid's completion
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n4; i += (int64_t)gridDim.x * 256)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// W13 row interleave for the prepack: destination row r of an expert's
// [2I, H] block <- source row (gate rows 0..I-1, up rows I..2I-1), groups of 32.
__global__ void w13_interleave_map_kernel(int32_t* map, int64_t I) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < 2 * I; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = r / 64, w = r % 64;
        map[r] = (int32_t)(w < 32 ? b * 32 + w : I + b * 32 + (w - 32));
    }
}

static cudaError_t launch_k(const void* fn, dim3 grid, dim3 block, size_t smem, bool pdl, cudaStream_t s,
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

}  // namespace fp4

using namespace fp4;

#define MOE_CHECK(cond, status, ...) \
    do {                             \
        if (!(cond)) {               \
            set_error(__VA_ARGS__);  \
            return (status);         \
        }                            \
    } while (0)

#define MOE_CUDA(call, what)                                                   \
    do {                                                                       \
        cudaError_t _e = (call);                                               \
        if (_e != cudaSuccess) {                                               \
            cudaGetLastError();                                                \
            set_error("%s: %s", what, cudaGetErrorString(_e));                 \
            return FP4_ERR_CUDA;                                               \
        }                                                                      \
    } while (0)

static bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

// ------------------------------------------------------------ prepack

extern "C" size_t fp4_moe_prepack_workspace_size(int64_t E, int64_t H, int64_t I) {
    (void)E;
    (void)H;
    if (I <= 0) return 4096;
    return 4096 + (size_t)a256(2 * I * 4);
}

extern "C" fp4_status fp4_moe_prepack_weights(const void* w13, const void* w2, int64_t E, int64_t H, int64_t I,
                                              void* w13_codes, void* w13_scales, float* w13_global, void* w2_codes,
                                              void* w2_scales, float* w2_global, void* ws, size_t wsb,
                                              void* stream) {
    MOE_CHECK(E > 0 && E <= kMaxExperts, FP4_ERR_SHAPE, "n_experts = %lld must be in [1, %d]", (long long)E,
              kMaxExperts);
    MOE_CHECK(H > 0 && H % 128 == 0 && I > 0 && I % 64 == 0, FP4_ERR_SHAPE,
              "hidden must be a positive multiple of 128 and inter of 64 (hidden %lld, inter %lld)", (long long)H,
              (long long)I);
    MOE_CHECK(w13 && w2 && w13_codes && w13_scales && w13_global && w2_codes && w2_scales && w2_global,
              FP4_ERR_INVALID_ARG, "null pointer argument");
    MOE_CHECK(al16(w13) && al16(w2) && al16(w13_codes) && al16(w13_scales) && al16(w2_codes) && al16(w2_scales) &&
                  ((uintptr_t)w13_global & 3) == 0 && ((uintptr_t)w2_global & 3) == 0,
              FP4_ERR_ALIGNMENT, "pointers must be 16-byte aligned (global scales 4-byte)");
    const size_t need = fp4_moe_prepack_workspace_size(E, H, I);
    MOE_CHECK(ws && wsb >= need && al16(ws), FP4_ERR_WORKSPACE, "workspace %zu bytes, need %zu", wsb, need);
    fp4_status st = check_arch();
    if (st != FP4_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* partials = static_cast<float*>(ws);
    int32_t* map = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + 4096);
    w13_interleave_map_kernel<<<(unsigned)((2 * I + 255) / 256), 256, 0, s>>>(map, I);
    MOE_CUDA(cudaGetLastError(), "interleave map launch");
    const size_t sc13 = (size_t)round_up(2 * I, 128) * sf_cols_padded(H, 16);
    const size_t sc2 = (size_t)round_up(H, 128) * sf_cols_padded(I, 16);
    for (int64_t e = 0; e < E; ++e) {
        for (int which = 0; which < 2; ++which) {
            QuantLaunch q;
            q.fmt = FP4_NVFP4;
            if (which == 0) {
                q.x = static_cast<const uint16_t*>(w13) + e * 2 * I * H;
                q.x_ld = H;
                q.rows = 2 * I;
                q.k = H;
                q.row_map = map;
                q.codes = static_cast<uint8_t*>(w13_codes) + e * 2 * I * (H / 2);
                q.scales = static_cast<uint8_t*>(w13_scales) + e * sc13;
                q.global_out = w13_global + e;
            } else {
                q.x = static_cast<const uint16_t*>(w2) + e * H * I;
                q.x_ld = I;
                q.rows = H;
                q.k = I;
                q.codes = static_cast<uint8_t*>(w2_codes) + e * H * (I / 2);
                q.scales = static_cast<uint8_t*>(w2_scales) + e * sc2;
                q.global_out = w2_global + e;
            }
            q.rows_pad = round_up(q.rows, 128);
            const int np = amax_partials_count(q.rows * q.k);
            MOE_CUDA(launch_amax_partials(q.x, q.rows * q.k, partials, np, false, s), "amax launch");
            q.sg_mode = SG_PARTIALS;
            q.partials = partials;
            q.n_partials = np;
            MOE_CUDA(launch_quant(q, s), "quantise launch");
        }
    }
    return FP4_OK;
}

// ------------------------------------------------------------ forward

extern "C" size_t fp4_moe_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return 0;
    return (size_t)moe_layout(T, H, I, E, k).total;
}

extern "C" int fp4_moe_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int64_t* offsets,
                                        int max_entries) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || !offsets) return 0;
    MoeLayout L = moe_layout(T, H, I, E, k);
    int n = 0;
    for (int i = 0; i < MS_PUBLIC_END && n < max_entries; ++i) offsets[n++] = L.off[i];
    if (n < max_entries) offsets[n++] = L.R;
    const int fused[] = {MS_F_H, MS_F_HCODES, MS_F_HSB, MS_F_SGH, MS_F_D, MS_F_ACODES, MS_F_ASB};
    for (int i = 0; i < 7 && n < max_entries; ++i) offsets[n++] = L.off[fused[i]];
    return n;
}

static int g_moe_policy = 0;  // fp4_set_moe_policy

extern "C" fp4_status fp4_set_moe_policy(int policy) {
    if (policy < 0 || policy > 2) {
        set_error("MoE policy %d not in 0..2", policy);
        return FP4_ERR_INVALID_ARG;
    }
    g_moe_policy = policy;
    return FP4_OK;
}

enum : unsigned { ST_ROUTE = 1u, ST_QUANT = 2u, ST_GEMM1 = 4u, ST_REQUANT = 8u, ST_GEMM2 = 16u, ST_ALL = 31u };

static fp4_status moe_run(const void* hidden, const float* logits, int64_t T, int64_t H, int64_t I, int64_t E,
                          int64_t k, int mode, const float* s13, const float* s2, const void* w13c,
                          const void* w13s, const float* w13g, const void* w2c, const void* w2s, const float* w2g,
                          void* out, void* ws, size_t wsb, unsigned mask, void* stream) {
    MOE_CHECK(T >= 0 && T < (1ll << 26), FP4_ERR_SHAPE, "tokens = %lld out of range", (long long)T);
    MOE_CHECK(E > 0 && E <= kMaxExperts, FP4_ERR_SHAPE, "n_experts = %lld must be in [1, %d]", (long long)E,
              kMaxExperts);
    MOE_CHECK(k > 0 && k <= E && k <= kMaxTopK, FP4_ERR_INVALID_ARG, "top_k = %lld must be in [1, min(E, %d)]",
              (long long)k, kMaxTopK);
    MOE_CHECK(H > 0 && H % 128 == 0 && I > 0 && I % 64 == 0, FP4_ERR_SHAPE,
              "hidden must be a positive multiple of 128 and inter of 64");
    MOE_CHECK(mode == FP4_SCALE_DYNAMIC || mode == FP4_SCALE_STATIC, FP4_ERR_INVALID_ARG, "unknown scale mode %d",
              mode);
    if (mode == FP4_SCALE_STATIC) {
        MOE_CHECK(s13 != nullptr && s2 != nullptr, FP4_ERR_MISSING_SCALE,
                  "static scale mode without per-expert activation scales (a weight-only checkpoint must use "
                  "FP4_SCALE_DYNAMIC)");
        MOE_CHECK(E <= kMaxStaticExperts, FP4_ERR_SHAPE, "static scale mode supports at most %d experts",
                  kMaxStaticExperts);
        for (int64_t e = 0; e < E; ++e)
            MOE_CHECK(isfinite(s13[e]) && s13[e] > 0.0f && isfinite(s2[e]) && s2[e] > 0.0f, FP4_ERR_INVALID_SCALE,
                      "static activation scale of expert %lld is not finite and > 0 (%g, %g)", (long long)e,
                      (double)s13[e], (double)s2[e]);
    }
    if (T == 0) return check_arch();
    MOE_CHECK(hidden && logits && w13c && w13s && w13g && w2c && w2s && w2g && out, FP4_ERR_INVALID_ARG,
              "null pointer argument");
    MOE_CHECK(al16(hidden) && al16(logits) && al16(w13c) && al16(w13s) && al16(w2c) && al16(w2s) && al16(out) &&
                  ((uintptr_t)w13g & 3) == 0 && ((uintptr_t)w2g & 3) == 0,
              FP4_ERR_ALIGNMENT, "pointers must be 16-byte aligned (global scales 4-byte)");
    const MoeLayout L = moe_layout(T, H, I, E, k);
    MOE_CHECK(ws && wsb >= (size_t)L.total && ((uintptr_t)ws & 255) == 0, FP4_ERR_WORKSPACE,
              "workspace %zu bytes, need %lld (256-byte aligned)", wsb, (long long)L.total);
    fp4_status st = check_arch();
    if (st != FP4_OK) return st;
    const DeviceInfo* d = current_device();
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t* b = static_cast<uint8_t*>(ws);
    auto at = [&](int slot) { return b + L.off[slot]; };
    int32_t* ids = (int32_t*)at(MS_IDS);
    float* wts = (float*)at(MS_WEIGHTS);
    int32_t* offsets = (int32_t*)at(MS_OFFSETS);
    int32_t* padded = (int32_t*)at(MS_PADDED);
    int32_t* row_src = (int32_t*)at(MS_ROW_SRC);
    uint8_t* a_codes = at(MS_A_CODES);
    uint8_t* a_scales = at(MS_A_SCALES);
    float* sg_a = (float*)at(MS_SG_A);
    uint16_t* h = (uint16_t*)at(MS_H);
    float* amax_h = (float*)at(MS_AMAX_H);
    float* sg_h = (float*)at(MS_SG_H);
    uint8_t* h_codes = at(MS_H_CODES);
    uint8_t* h_scales = at(MS_H_SCALES);
    float* y = (float*)at(MS_Y);
    uint32_t* bitmap = (uint32_t*)at(MS_BITMAP);
    int32_t* wprefix = (int32_t*)at(MS_WPREFIX);
    int32_t* tile_expert = (int32_t*)at(MS_TILE_EXPERT);
    int32_t* n_ptiles = (int32_t*)at(MS_NPTILES);
    int32_t* row_valid_end = (int32_t*)at(MS_ROW_VALID_END);
    int32_t* row_tok = (int32_t*)at(MS_ROW_TOK);
    float* partials = (float*)at(MS_PARTIALS);
    float* st13 = (float*)at(MS_STATIC13);
    float* st2 = (float*)at(MS_STATIC2);
    const bool is_static = mode == FP4_SCALE_STATIC;
    const bool full = (mask & ST_ALL) == ST_ALL;
    // A few tokens per expert (at most 16 on average): the grouped GEMMs swap
    // their operands, so the expert's weight rows fill the 128-row MMA side and
    // its tokens a 32-column one, instead of padding the tokens to 128 rows.
    const bool swapped = T * k <= 16 * E;
    // the whole pipeline for a handful of tokens: one launch prepares it all
    const bool small_prep = full && swapped && T <= kPrepMaxTokens;
    bool pdl = false;  // first launch of the call waits for everything before it
    const int per_lane = (int)((E + 31) / 32);

    // the one launch where it is faster than the chain (automatic), or whenever it applies (policy 2)
    const bool fused = g_moe_policy == 2 || (g_moe_policy == 0 && T <= kFusedAutoMaxT);
    if (full && fused && moe_fused_supported(T, H, I, E, k)) {
        // a few tokens: the whole layer in one launch (after a memset of its counters)
        FusedMoeLaunch F;
        F.hidden = static_cast<const uint16_t*>(hidden);
        F.logits = logits;
        F.T = T, F.H = H, F.I = I, F.E = E, F.k = k;
        F.is_static = is_static ? 1 : 0;
        F.w13_codes = static_cast<const uint8_t*>(w13c);
        F.w13_scales = static_cast<const uint8_t*>(w13s);
        F.w13_global = w13g;
        F.w2_codes = static_cast<const uint8_t*>(w2c);
        F.w2_scales = static_cast<const uint8_t*>(w2s);
        F.w2_global = w2g;
        F.out = static_cast<uint16_t*>(out);
        F.ids = ids;
        F.weights = wts;
        F.sg_a = sg_a;
        F.zeroed = (uint32_t*)at(MS_F_ZERO);
        F.h = (uint16_t*)at(MS_F_H);
        F.a_codes = at(MS_F_ACODES);
        F.a_sbytes = at(MS_F_ASB);
        F.h_codes = at(MS_F_HCODES);
        F.h_sbytes = at(MS_F_HSB);
        F.sg_h = (float*)at(MS_F_SGH);
        F.d = (float*)at(MS_F_D);
        StaticScales sc;
        memset(&sc, 0, sizeof(sc));
        if (is_static)
            for (int64_t e = 0; e < E; ++e) sc.s13[e] = s13[e], sc.s2[e] = s2[e];
        MOE_CUDA(launch_moe_fused(F, sc, s), "fused MoE launch");
        return FP4_OK;
    }

    if (small_prep) {
        PrepArgs pa;
        pa.logits = logits;
        pa.hidden = static_cast<const uint16_t*>(hidden);
        pa.T = T;
        pa.H = H;
        pa.E = (int)E;
        pa.k = (int)k;
        pa.ids = ids;
        pa.weights = wts;
        pa.offsets = offsets;
        pa.padded = padded;
        pa.n_ptiles = n_ptiles;
        pa.tile_expert = tile_expert;
        pa.row_valid_end = row_valid_end;
        pa.row_src = row_src;
        pa.row_tok = row_tok;
        pa.codes = a_codes;
        pa.scales = a_scales;
        pa.sg_out = sg_a;
        pa.has_static = is_static ? 1 : 0;
        pa.dispatch_inline = T <= kPrepInlineTokens ? 1 : 0;
        pa.slot_row = (int32_t*)at(MS_SLOT_ROW);
        pa.static13_out = st13;
        pa.static2_out = st2;
        pa.amax_h = amax_h;
        pa.y = y;
        pa.y_elems = 0;  // nothing to clear: GEMM2 writes every slot's row
        // the hidden abs-max in slices of 2048 16-byte vectors, one CTA each
        pa.amax_part = partials;
        pa.n_amax_ctas = (!is_static && !pa.dispatch_inline)
                             ? (int)std::min<int64_t>(32, std::max<int64_t>(1, (T * H / 8 + 2047) / 2048))
                             : 0;
        StaticScales sc;
        memset(&sc, 0, sizeof(sc));
        if (is_static)
            for (int64_t e = 0; e < E; ++e) sc.s13[e] = s13[e], sc.s2[e] = s2[e];
        pa.mark_pad_rows = 1;    // the swapped GEMMs never read the padding rows' scales
        pa.zero_pad_scales = 0;
        const int zero_blocks = pa.n_amax_ctas;
        void* args[] = {(void*)&pa, (void*)&sc};
        const void* fn = per_lane <= 4    ? (const void*)moe_prep_small_kernel<4>
                         : per_lane <= 8  ? (const void*)moe_prep_small_kernel<8>
                         : per_lane <= 16 ? (const void*)moe_prep_small_kernel<16>
                                          : (const void*)moe_prep_small_kernel<32>;
        MOE_CUDA(launch_k(fn, dim3(1 + zero_blocks), dim3(1024), 0, pdl, s, args), "prepare launch");
        pdl = true;
        if (!pa.dispatch_inline) {
            const int64_t items = (is_static ? T * k : T) * sf_cols_padded(H, 16);
            const int64_t db = std::min<int64_t>((items + 255) / 256, (int64_t)d->sm_count * 4);
            MOE_CUDA(launch_k((const void*)moe_dispatch_kernel, dim3((unsigned)db), dim3(256), 0, pdl, s, args),
                     "dispatch launch");
        }
    }

    // 1. route (+ zeroing of y and amax_h when the whole pipeline runs)
    if ((mask & ST_ROUTE) && !small_prep) {
        RouteArgs ra;
        ra.logits = logits;
        ra.T = T;
        ra.E = (int)E;
        ra.k = (int)k;
        ra.ids = ids;
        ra.weights = wts;
        ra.bitmap = bitmap;
        ra.W = L.W;
        ra.y = y;
        ra.y_elems = 0;  // nothing to clear: GEMM2 writes every slot's row
        ra.amax_h = amax_h;
        ra.route_blocks = (int)((T + 31) / 32);  // one CTA (32 warps) per 32 tokens = one bitmap word
        ra.has_static = is_static ? 1 : 0;
        ra.static13_out = st13;
        ra.static2_out = st2;
        ra.zero_outputs = full ? 1 : 0;
        StaticScales sc;
        memset(&sc, 0, sizeof(sc));
        if (is_static)
            for (int64_t e = 0; e < E; ++e) sc.s13[e] = s13[e], sc.s2[e] = s2[e];
        const int zero_blocks = 0;
        void* args[] = {(void*)&ra, (void*)&sc};
        const void* fn = per_lane <= 4    ? (const void*)moe_route_kernel<4>
                         : per_lane <= 8  ? (const void*)moe_route_kernel<8>
                         : per_lane <= 16 ? (const void*)moe_route_kernel<16>
                                          : (const void*)moe_route_kernel<32>;
        MOE_CUDA(launch_k(fn, dim3(ra.route_blocks + zero_blocks), dim3(1024), (size_t)E * 4, pdl, s, args),
                 "route launch");
        pdl = true;
        ScanArgs sa;
        sa.bitmap = bitmap;
        sa.wprefix = wprefix;
        sa.ids = ids;
        sa.T = T;
        sa.W = L.W;
        sa.E = (int)E;
        sa.k = (int)k;
        sa.offsets = offsets;
        sa.padded = padded;
        sa.n_ptiles = n_ptiles;
        sa.tile_expert = tile_expert;
        sa.row_valid_end = row_valid_end;
        sa.row_src = row_src;
        sa.row_tok = row_tok;
        sa.slot_row = (int32_t*)at(MS_SLOT_ROW);
        void* sargs[] = {(void*)&sa};
        MOE_CUDA(launch_k((const void*)moe_scan_kernel, dim3(1), dim3(1024), 0, pdl, s, sargs), "scan launch");
        const int64_t ab = std::min<int64_t>((T * k + 255) / 256, (int64_t)d->sm_count * 8);
        MOE_CUDA(launch_k((const void*)moe_assign_kernel, dim3((unsigned)ab), dim3(256), 0, pdl, s, sargs),
                 "assign launch");
    }
    // 2-3. hidden amax (dynamic) and quantise into expert-sorted padded rows
    if ((mask & ST_QUANT) && !small_prep) {
        QuantLaunch q;
        q.fmt = FP4_NVFP4;
        q.x = static_cast<const uint16_t*>(hidden);
        q.x_ld = H;
        q.rows = L.R;
        q.rows_pad = L.R;
        q.k = H;
        q.row_map = row_tok;
        q.codes = a_codes;
        q.scales = a_scales;
        q.rows_dev = nullptr;
        q.pdl = pdl;
        q.tile_expert = tile_expert;
        q.n_experts = (int)E;
        if (!is_static) {
            // one per-tensor scale: the abs-max in partials, then each token row
            // quantised once into the rows of its k routing slots; the tiles'
            // padding rows get zero scale bytes (GEMM1 reads them)
            const int np = amax_partials_count(T * H);
            MOE_CUDA(launch_amax_partials(q.x, T * H, partials, np, pdl, s), "amax launch");
            PrepArgs pa;
            memset(&pa, 0, sizeof(pa));
            pa.hidden = static_cast<const uint16_t*>(hidden);
            pa.T = T;
            pa.H = H;
            pa.E = (int)E;
            pa.k = (int)k;
            pa.ids = ids;
            pa.n_ptiles = n_ptiles;
            pa.row_valid_end = row_valid_end;
            pa.row_src = row_src;
            pa.row_tok = row_tok;
            pa.slot_row = (int32_t*)at(MS_SLOT_ROW);
            pa.codes = a_codes;
            pa.scales = a_scales;
            pa.sg_out = sg_a;
            pa.amax_part = partials;
            pa.n_amax_ctas = np;
            pa.mark_pad_rows = 0;  // the scan marked them
            pa.zero_pad_scales = 1;
            StaticScales sc;
            memset(&sc, 0, sizeof(sc));
            void* dargs[] = {(void*)&pa, (void*)&sc};
            const int64_t items = T * sf_cols_padded(H, 16);
            const int64_t db = std::min<int64_t>((items + 255) / 256, (int64_t)d->sm_count * 4);
            MOE_CUDA(launch_k((const void*)moe_dispatch_kernel, dim3((unsigned)db), dim3(256), 0, true, s, dargs),
                     "dispatch launch");
        } else {
            q.sg_mode = SG_EXPERT_TABLE;
            q.table = st13;
            // rows beyond the padded total are skipped: their count is on the device
            q.rows_dev = padded + E;
            MOE_CUDA(launch_quant(q, s), "quantise launch");
        }
        pdl = true;
    }
    // 4. GEMM1 + SiLU * up + per-expert amax of h
    if (mask & ST_GEMM1) {
        if (!full) {
            float4* z = reinterpret_cast<float4*>(amax_h);
            int64_t n4 = (E + 3) / 4;
            void* zargs[] = {(void*)&z, (void*)&n4};
            MOE_CUDA(launch_k((const void*)zero_kernel, dim3(1), dim3(256), 0, pdl, s, zargs), "zero launch");
            pdl = true;
        }
        GemmLaunch g;
        g.fmt = FP4_NVFP4;
        if (swapped) {
            g.epi = EPI_SWIGLU_T;
            g.bn = 32;
            g.p_codes = static_cast<const uint8_t*>(w13c);
            g.p_scales = static_cast<const uint8_t*>(w13s);
            g.p_rows = E * 2 * I;
            g.p_rows_valid = 2 * I;
            g.q_codes = a_codes;
            g.q_scales = a_scales;
            g.q_rows = L.R;
            g.q_rows_valid = L.R;
            g.p_global = w13g;
            g.q_global = is_static ? st13 : sg_a;
            g.q_global_per_expert = is_static;
        } else {
            g.epi = EPI_SWIGLU;
            // the tile width must divide the expert's 2I rows (tiles never straddle
            // experts); 128 keeps two TMEM accumulators, so the SwiGLU epilogue of
            // one tile overlaps the next tile's MMAs (with 256 there is one)
            g.bn = (T * k >= 4 * E * 64 && (2 * I) % 128 == 0) ? 128 : 64;
            g.p_codes = a_codes;
            g.p_scales = a_scales;
            g.p_rows = L.R;
            g.q_codes = static_cast<const uint8_t*>(w13c);
            g.q_scales = static_cast<const uint8_t*>(w13s);
            g.q_rows = E * 2 * I;
            g.q_rows_valid = 2 * I;
            g.p_global = is_static ? st13 : sg_a;
            g.p_global_per_expert = is_static;
            g.q_global = w13g;
        }
        g.k = H;
        g.out = h;
        g.ldo = I;
        g.grouped = true;
        g.n_experts = (int)E;
        g.tile_expert = tile_expert;
        g.n_ptiles_dev = n_ptiles;
        g.row_valid_end = row_valid_end;
        g.amax_out = amax_h;
        g.pdl = pdl;
        MOE_CUDA(launch_gemm(g, s), "GEMM1 launch");
        pdl = true;
    }
    // 5. requantise h per expert
    if (mask & ST_REQUANT) {
        QuantLaunch q;
        q.fmt = FP4_NVFP4;
        q.x = h;
        q.x_ld = I;
        q.rows = L.R;
        q.rows_pad = L.R;
        q.k = I;
        q.row_map = row_tok;
        q.row_map_is_mask = true;
        // the swapped GEMM2 discards padding columns: their scale bytes need
        // not be zeroed when the whole pipeline runs, and only each tile's
        // real rows are walked (with many tokens per expert the padded walk
        // of the generic kernel is faster: one full tile per CTA leaves each
        // thread a long serial chain, 97 us against 41 us at T = 4096)
        q.skip_masked_rows = full && swapped;
        q.tile_rows_end = row_valid_end;
        q.n_tiles_dev = n_ptiles;
        q.codes = h_codes;
        q.scales = h_scales;
        q.tile_expert = tile_expert;
        q.n_experts = (int)E;
        q.rows_dev = padded + E;
        q.pdl = pdl;
        if (!is_static) {
            q.sg_mode = SG_EXPERT_AMAX;
            q.table = amax_h;
            q.expert_sg_out = sg_h;
        } else {
            q.sg_mode = SG_EXPERT_TABLE;
            q.table = st2;
        }
        MOE_CUDA(launch_quant(q, s), "requantise launch");
        pdl = true;
    }
    // 6. GEMM2 into one fp32 row per routing slot, then the top-k sum in slot order -> bf16
    if (mask & ST_GEMM2) {
        GemmLaunch g;
        g.fmt = FP4_NVFP4;
        if (swapped) {
            g.epi = EPI_DSLOT_T;
            g.bn = 32;
            g.p_codes = static_cast<const uint8_t*>(w2c);
            g.p_scales = static_cast<const uint8_t*>(w2s);
            g.p_rows = E * H;
            g.p_rows_valid = H;
            g.q_codes = h_codes;
            g.q_scales = h_scales;
            g.q_rows = L.R;
            g.q_rows_valid = L.R;
            g.p_global = w2g;
            g.q_global = is_static ? st2 : sg_h;
            g.q_global_per_expert = true;
        } else {
            g.epi = EPI_DSLOT;
            // the tile width must divide H (output columns of one token row); the
            // fp32 epilogue keeps at most 64 columns per warp in registers
            g.bn = (T * k >= 4 * E * 64 && H % 128 == 0) ? 128 : 64;
            g.p_codes = h_codes;
            g.p_scales = h_scales;
            g.p_rows = L.R;
            g.q_codes = static_cast<const uint8_t*>(w2c);
            g.q_scales = static_cast<const uint8_t*>(w2s);
            g.q_rows = E * H;
            g.q_rows_valid = H;
            g.p_global = is_static ? st2 : sg_h;
            g.p_global_per_expert = true;
            g.q_global = w2g;
        }
        g.k = I;
        g.out = y;
        g.ldo = H;
        g.grouped = true;
        g.n_experts = (int)E;
        g.tile_expert = tile_expert;
        g.n_ptiles_dev = n_ptiles;
        g.row_valid_end = row_valid_end;
        g.pdl = pdl;
        MOE_CUDA(launch_gemm(g, s), "GEMM2 launch");
        const float4* d4 = reinterpret_cast<const float4*>(y);
        const float* wv = wts;
        const int32_t* sr = (const int32_t*)at(MS_SLOT_ROW);
        uint2* o2 = reinterpret_cast<uint2*>(out);
        int64_t TT = T, h4 = H / 4;
        int kk = (int)k;
        void* fargs[] = {(void*)&d4, (void*)&wv, (void*)&sr, (void*)&TT, (void*)&kk, (void*)&h4, (void*)&o2};
        int64_t fb = std::min<int64_t>((T * h4 + 255) / 256, (int64_t)d->sm_count * 8);
        MOE_CUDA(launch_k((const void*)moe_combine_kernel, dim3((unsigned)fb), dim3(256), 0, true, s, fargs),
                 "combine launch");
    }
    return FP4_OK;
}

extern "C" fp4_status fp4_moe_grouped(const void* hidden, const float* logits, int64_t T, int64_t H, int64_t I,
                                      int64_t E, int64_t k, int mode, const float* s13, const float* s2,
                                      const void* w13c, const void* w13s, const float* w13g, const void* w2c,
                                      const void* w2s, const float* w2g, void* out, void* ws, size_t wsb,
                                      void* stream) {
    return moe_run(hidden, logits, T, H, I, E, k, mode, s13, s2, w13c, w13s, w13g, w2c, w2s, w2g, out, ws, wsb,
                   ST_ALL, stream);
}

extern "C" fp4_status fp4_moe_grouped_stages(const void* hidden, const float* logits, int64_t T, int64_t H,
                                             int64_t I, int64_t E, int64_t k, int mode, const float* s13,
                                             const float* s2, const void* w13c, const void* w13s, const float* w13g,
                                             const void* w2c, const void* w2s, const float* w2g, void* out, void* ws,
                                             size_t wsb, unsigned mask, void* stream) {
    return moe_run(hidden, logits, T, H, I, E, k, mode, s13, s2, w13c, w13s, w13g, w2c, w2s, w2g, out, ws, wsb,
                   mask & ST_ALL, stream);
}
