// moe_common.cuh -- pieces shared by the MoE launch chain (moe.cu) and the
// one-launch MoE for a few tokens (moe_fused.cu): limits, the static-scale
// kernel parameter and the warp-cooperative router.
#pragma once

#include <math.h>

#include "common.cuh"

namespace fp4 {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxStaticExperts = 256;

// Per-expert static activation scales, passed by value as a kernel parameter.
struct StaticScales {
    float s13[kMaxStaticExperts];
    float s2[kMaxStaticExperts];
};

// The one-launch MoE for a few tokens (moe_fused.cu).
constexpr int kFusedMaxT = 16;                        // tokens
constexpr int kFusedAutoMaxT = 16;                    // tokens up to which fp4_moe_grouped takes it by default
constexpr int kFusedMaxTopK = 8;
constexpr int kFusedMaxSlots = kFusedMaxT * kFusedMaxTopK;
constexpr int kFusedMaxK = 2048;                      // H and I (the two GEMMs' K)
constexpr int kFusedMaxE = 256;                       // experts
constexpr int kFusedMaxOutTiles = 32;                 // H / 128
constexpr int kFusedZeroedBytes = 2048;               // counters + h amax, cleared per call

struct FusedMoeLaunch {
    const uint16_t* hidden;
    const float* logits;
    int64_t T, H, I, E, k;
    int is_static;
    const uint8_t* w13_codes;
    const uint8_t* w13_scales;
    const float* w13_global;
    const uint8_t* w2_codes;
    const uint8_t* w2_scales;
    const float* w2_global;
    uint16_t* out;
    int32_t* ids;
    float* weights;
    float* sg_a;
    uint32_t* zeroed;  // kFusedZeroedBytes, cleared by the launcher
    uint16_t* h;
    uint8_t* a_codes;
    uint8_t* a_sbytes;
    uint8_t* h_codes;
    uint8_t* h_sbytes;
    float* sg_h;
    float* d;
};

// The shapes the one-launch MoE takes (else the launch chain runs).
bool moe_fused_supported(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k);
// One memset (the counters) and one cooperative kernel launch.
cudaError_t launch_moe_fused(const FusedMoeLaunch& L, const StaticScales& st, cudaStream_t s);

// Order-preserving 32-bit key of a logit: a larger float has a larger key.
// -0 ranks with +0 (the two compare equal), and a NaN ranks below every
// number (a stable descending sort of the logits puts it last); key 0 is
// left for "no candidate".
__device__ __forceinline__ uint32_t route_key(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 1u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The logit of a key (route_key's inverse on numbers).
__device__ __forceinline__ float route_val(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Warp-cooperative top-k over one token's logits, lane l holding logits
// l, 32 + l, 64 + l, ... in v (ignored past E); ties go to the lower expert
// index.  Lane j < k returns the j-th selection and its weight
// exp(l_j - l_max) / sum over the selection.  Each round takes the largest
// key with one warp max-reduction and, among the lanes holding it, the
// lowest expert index with one min-reduction (a lane's own candidate is
// its first register with its largest key, so its lowest index).
template <int PER_LANE>
__device__ __forceinline__ void topk_regs(const float (&v)[PER_LANE], int E, int k, int lane, int& my_e,
                                          float& my_w) {
    uint32_t key[PER_LANE];
#pragma unroll
    for (int q = 0; q < PER_LANE; ++q) key[q] = q * 32 + lane < E ? route_key(v[q]) : 0u;
    float v0 = 0.0f, sum = 0.0f, mine = 0.0f;
    my_e = 0;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = key[0], bq = 0;
#pragma unroll
        for (int q = 1; q < PER_LANE; ++q)
            if (key[q] > bk) {
                bk = key[q];
                bq = (uint32_t)q;
            }
        const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const uint32_t be = __reduce_min_sync(0xFFFFFFFFu, bk == mk ? bq * 32u + (uint32_t)lane : 0xFFFFFFFFu);
        if ((be & 31u) == (uint32_t)lane) {
#pragma unroll
            for (int q = 0; q < PER_LANE; ++q)
                if ((uint32_t)q == (be >> 5)) key[q] = 0u;
        }
        const float bv = route_val(mk);
        if (j == 0) v0 = bv;
        const float ex = expf(bv - v0);
        sum += ex;
        if (lane == j) {
            my_e = (int)be;
            mine = ex;
        }
    }
    my_w = __fdiv_rn(mine, sum);
}

// The same, loading the token's logits row.
template <int PER_LANE>
__device__ __forceinline__ void topk_token(const float* row, int E, int k, int lane, int& my_e, float& my_w) {
    float v[PER_LANE];
#pragma unroll
    for (int q = 0; q < PER_LANE; ++q) {
        const int e = q * 32 + lane;
        v[q] = e < E ? row[e] : -INFINITY;
    }
    topk_regs<PER_LANE>(v, E, k, lane, my_e, my_w);
}

}  // namespace fp4
