// internal.h -- host-side interface between the libfp4 translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4.h"

namespace fp4 {

struct DeviceInfo {
    int device = -1;
    int cc = 0;          // compute capability, major*10 + minor
    int sm_count = 0;
    int l2_bytes = 0;
    uint32_t* err_word = nullptr;  // device error flags (file-scope __device__ word)
};

// Cached per-device facts for the current device; nullptr on a CUDA error.
const DeviceInfo* current_device();

// Nanoseconds a device-side wait may spin before giving up.
uint64_t wait_limit_ns();

// Opt `fn` in to `bytes` of dynamic shared memory on the current device, once
// per device; `done` is the caller's per-kernel mask of devices already set.
cudaError_t set_smem_attr_once(const void* fn, int bytes, uint64_t& done);

void set_error(const char* fmt, ...);

// FP4_OK if the current device is sm_103 (honours fp4_set_arch_override).
fp4_status check_arch();

// ------------------------------------------------------------- quantiser

// How each row's global scale s_g is obtained.
enum SgMode : int {
    SG_PARTIALS = 0,      // dynamic: amax = max(partials[0..n)), s_g = amax / 2688
    SG_STATIC = 1,        // s_g = static_scale
    SG_EXPERT_TABLE = 2,  // s_g = table[tile_expert[row / 128]]
    SG_EXPERT_AMAX = 3,   // s_g = amax[tile_expert[row / 128]] / 2688
};

struct QuantLaunch {
    int fmt = FP4_NVFP4;
    const uint16_t* x = nullptr;  // source rows (bf16 bits)
    int64_t x_ld = 0;             // source row stride, elements
    int64_t rows = 0;             // destination rows written with codes
    int64_t rows_pad = 0;         // destination rows whose scales are written (>= rows, multiple of 128)
    int64_t k = 0;
    const int32_t* row_map = nullptr;  // dest row -> source row (-1: zero row); nullptr = identity
    bool row_map_is_mask = false;      // row_map[r] >= 0 only marks row r as real (source row = r)
    bool skip_masked_rows = false;     // rows the map marks absent are left untouched (scale bytes too)
    // with skip_masked_rows and an expert scale: the real rows are those of each
    // 128-row tile t < *n_tiles_dev below tile_rows_end[t] (the rest are skipped)
    const int32_t* tile_rows_end = nullptr;
    const int32_t* n_tiles_dev = nullptr;
    uint8_t* codes = nullptr;
    uint8_t* scales = nullptr;
    int sg_mode = SG_STATIC;
    float static_scale = 0.f;
    const float* partials = nullptr;
    int n_partials = 0;
    const float* table = nullptr;       // SG_EXPERT_TABLE / SG_EXPERT_AMAX source, per expert
    const int32_t* tile_expert = nullptr;
    float* global_out = nullptr;        // SG_PARTIALS / SG_STATIC: s_g written here
    float* expert_sg_out = nullptr;     // SG_EXPERT_AMAX: s_g[e] written here (n_experts entries)
    int n_experts = 0;
    const int32_t* rows_dev = nullptr;  // optional device row count bound (grouped): rows beyond are skipped
    bool pdl = false;
    // x was complete before the grid this launch depends on started (that grid
    // writes only the partials): quant_nv_kernel may load its first rows before
    // the dependency wait
    bool x_before_wait = false;
};

int amax_partials_count(int64_t n_elems);
cudaError_t launch_amax_partials(const uint16_t* x, int64_t n_elems, float* partials, int n_part, bool pdl,
                                 cudaStream_t s);
cudaError_t launch_quant(const QuantLaunch& q, cudaStream_t s);

// ------------------------------------------------------------------ GEMM

enum Epi : int {
    EPI_BF16 = 0,       // out[p][q] = bf16(alpha * acc)            (row-major, P = activations)
    EPI_BF16_T = 1,     // out[q][p] = bf16(alpha * acc)            (P = weights, swap-AB)
    EPI_PARTIAL_T = 2,  // part[split][q][p] = acc (fp32, alpha applied by the reduction)
    EPI_SWIGLU = 3,     // grouped: h[p][f] = bf16(SiLU(gate) * up), amax per expert
    EPI_PARTIAL = 5,    // part[split][p][q] = acc (fp32, P = activations; alpha applied by the reduction)
    // grouped with the operands swapped (P = an expert's weight rows, Q = 32-row
    // tiles of its tokens), for a few tokens per expert:
    EPI_SWIGLU_T = 6,   // h[q][f] = bf16(SiLU(gate) * up), amax per expert
    // grouped GEMM2 outputs per routing slot (token * top_k + j), fp32, summed
    // in slot order by a separate combine (same bits every run):
    EPI_DSLOT = 8,      // d[p][q] = alpha * acc (fp32, TMA stores; P = expert-sorted token rows)
    EPI_DSLOT_T = 9,    // d[q][p] = alpha * acc (swapped: P = an expert's weight rows)
};

// GemmLaunch::fmt for the 8-bit-container MX formats (MXFP8 / MXFP6; codes
// one byte per element, UE8M0 scales per 32), beside FP4_NVFP4 / FP4_MXFP4.
constexpr int FMT_MX8 = 2;

struct GemmLaunch {
    int fmt = FP4_NVFP4;
    int p_type = 0, q_type = 0;   // FMT_MX8: element type codes of P and Q (kind::mxf8f6f4 descriptor)
    int epi = EPI_BF16;
    int bn = 256;                 // Q tile rows (MMA N): 32, 64, 128 or 256
    // operand P (MMA A, 128-row tiles) and Q (MMA B, bn-row tiles), both K-major
    const uint8_t* p_codes = nullptr;
    const uint8_t* p_scales = nullptr;
    int64_t p_rows = 0;           // rows of the P tensor (TMA extent)
    const uint8_t* q_codes = nullptr;
    const uint8_t* q_scales = nullptr;
    int64_t q_rows = 0;           // rows of the Q tensor (all experts when grouped)
    int64_t q_rows_valid = 0;     // valid Q rows per tile group (per expert when grouped)
    int64_t k = 0;
    const float* p_global = nullptr;  // NVFP4 global scale(s) of P (per expert when grouped && p_global_per_expert)
    const float* q_global = nullptr;  // NVFP4 global scale(s) of Q (per expert when grouped)
    bool p_global_per_expert = false;
    bool q_global_per_expert = false;  // EPI_SWIGLU_T / EPI_DSLOT_T: Q (tokens) scale per expert
    // output
    void* out = nullptr;
    int64_t ldo = 0;
    int64_t p_rows_valid = 0;     // rows of P that are real (dense)
    int splits = 1;
    // grouped (MoE).  The token side is the P operand, or the Q operand with
    // the swapped epilogues (EPI_SWIGLU_T, EPI_DSLOT_T: P = weights, whose
    // per-expert row count is p_rows_valid); the tables below always describe
    // the token rows, in 128-row tiles.
    bool grouped = false;
    int n_experts = 0;
    const int32_t* tile_expert = nullptr;   // expert of each 128-row token tile
    const int32_t* n_ptiles_dev = nullptr;  // number of token tiles (device)
    const int32_t* row_valid_end = nullptr; // per token tile: first padded row index (exclusive end of real rows)
    float* amax_out = nullptr;              // EPI_SWIGLU: per-expert amax of h (as uint bits, atomicMax)
    int max_ctas = 0;                       // 0 = one per SM
    bool mc = false;                        // dense EPI_BF16, bn 256, an even number of 128-row P tiles:
                                            // clusters of two CTAs sharing each Q tile (TMA multicast)
    bool pdl = false;
    // Operand tiles that do not depend on the preceding kernel (the weights):
    // their producer starts loading before the programmatic-dependency wait,
    // overlapping the tail of the activation quantiser.  Non-grouped only.
    bool early_p = false;
    bool early_q = false;
};

// K block of the one-CTA GEMM pipeline: bytes of packed codes per row and
// stage (128: 256 FP4 elements, 128-byte swizzle; 64: 128 elements, 64-byte
// swizzle).  Each stage carries fixed costs (barrier round trips, scale
// stores, the MMA thread's waits), which the 64-byte block pays twice as
// often; 128 measured faster on the 8192 x 14336 x 4096 prefill.
constexpr int GEMM_KB_BYTES = 128;
int64_t gemm_k_blocks(int64_t k);  // K blocks of the one-CTA GEMM

// Small-M linear in one launch (decode_fused.cu): quantises the m <= 8 bf16
// activation rows in the kernel and streams the weights, one CTA per 128
// weight rows, bf16 out [m][n].
constexpr int kDecodeFusedMaxM = 8;
// rows up to which the automatic policy takes the fused kernel: on the
// 14336 x 4096 decode it is faster than the quantise + GEMM launches at every
// m <= 8 (about 5 us at m = 1, 2 us at m = 8); the in-kernel quantisation of
// every row by every CTA grows with m, so more rows go to the launch chain
constexpr int kDecodeFusedAutoMaxM = 8;
constexpr int64_t kDecodeFusedMaxK = 8192;
cudaError_t launch_decode_fused(int fmt, const uint16_t* x, int m, int64_t n, int64_t k, const uint8_t* w_codes,
                                const uint8_t* w_scales, const float* w_global, int dynamic, float static_scale,
                                float* a_global_out, uint16_t* out, bool pdl, cudaStream_t s);
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s);
// CTA-pair variant (EPI_BF16 only): 256 x 256 tiles on clusters of two CTAs.
cudaError_t launch_gemm_pair(const GemmLaunch& g, cudaStream_t s);
cudaError_t launch_splitk_reduce(const float* part, int splits, int64_t m, int64_t n, const float* ga,
                                 const float* gw, bool mx, uint16_t* out, bool pdl, cudaStream_t s);

}  // namespace fp4
