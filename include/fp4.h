/*
 * fp4.h -- C ABI of libfp4.so: block-scaled FP4 (NVFP4 / MXFP4) linear layer
 * and NVFP4 fused-MoE layer on one GB300 GPU (sm_103a).
 *
 * Formats ("vLLM on DGX Spark: technical report", section 6.1 "NVFP4 format"
 * and section 6.4 "NVFP4 vs MXFP4"):
 *   NVFP4: E2M1 elements {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6} packed two
 *          per byte, one FP8-E4M3 block scale per 16 contiguous elements along
 *          K, one fp32 global scale per tensor; value = element x block scale
 *          x global scale.
 *   MXFP4: E2M1 elements, one E8M0 (power-of-two) scale per 32 elements along
 *          K, no global scale.
 * The GEMM dequantises by alpha = weight global scale x activation global
 * scale ("GLM-5.3-Flash on vLLM, on GB10", the opening account of the MoE
 * activation-scale fault: each expert's alpha is weight_scale_2 x
 * input_scale).  All global scales in this ABI use that dequantisation
 * convention: s_g = amax / (6 x 448) for a dynamic scale.
 *
 * Memory layouts (all device memory unless stated otherwise):
 *   bf16 tensors   row-major, contiguous, 16-byte aligned base.
 *   codes          [rows][k/2] bytes, row-major; element 2j of a row is the low
 *                  nibble of byte j.  16-byte aligned base.
 *   scales         "MMA layout": rows padded to a multiple of 128, scale
 *                  columns padded to whole 256-element K tiles (16 NVFP4 or 8
 *                  MXFP4 columns per tile).  Atoms of 128 rows x 4 scale
 *                  columns = 512 bytes; inside an atom row r is at byte
 *                  (r % 32) * 16 + (r / 32) * 4 and scale column j at + (j %
 *                  4); atoms are ordered by 128-row tile, then by K.  Padding
 *                  bytes are written as 0 by the quantisers.  Size:
 *                  fp4_scales_bytes().  16-byte aligned base.
 *   global scale   one fp32 in device memory (per expert for the MoE).
 *
 * Shapes: k must be a positive multiple of 32 (16-byte rows of packed codes);
 * n must be a multiple of 8 (16-byte output rows); rows / m / T may be 0 (the
 * call then returns FP4_OK and launches nothing).  Row counts and n must be
 * below 2^31.
 *
 * Ownership: the caller allocates every buffer, including the workspace, and
 * keeps them alive until the work on `stream` has finished.  The library does
 * not allocate device memory, does not synchronise and never falls back to
 * another implementation.  `stream` is a cudaStream_t (NULL = legacy default
 * stream).  Calls that share a workspace must not overlap on the GPU.
 *
 * Errors: every argument that can be checked on the host is checked before
 * any launch; on failure the call returns the status, writes nothing and sets
 * a thread-local message (fp4_last_error_message).  A device that is not
 * sm_103 gives FP4_ERR_UNSUPPORTED_ARCH (loudly, never a trap and never a
 * silent result).  Launch failures give FP4_ERR_CUDA.  Kernels never trap:
 * every wait is bounded, and a wait that gives up records a device-side flag
 * that fp4_device_status() reports as FP4_ERR_DEVICE_TIMEOUT.
 */
#ifndef FP4_H
#define FP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP4_ABI_VERSION 1

typedef enum {
    FP4_OK = 0,
    FP4_ERR_INVALID_ARG = 1,      /* null pointer, bad enum, bad top_k, ... */
    FP4_ERR_SHAPE = 2,            /* k % 32, n % 8, negative or too-large sizes */
    FP4_ERR_ALIGNMENT = 3,        /* a pointer is not 16-byte (fp32: 4-byte) aligned */
    FP4_ERR_UNSUPPORTED_ARCH = 4, /* current device is not sm_103 */
    FP4_ERR_MISSING_SCALE = 5,    /* static scale mode without the scales */
    FP4_ERR_INVALID_SCALE = 6,    /* static scale <= 0, NaN or infinite */
    FP4_ERR_WORKSPACE = 7,        /* workspace missing or smaller than required */
    FP4_ERR_CUDA = 8,             /* a CUDA runtime call or launch failed */
    FP4_ERR_DEVICE_TIMEOUT = 9    /* a kernel's bounded wait gave up */
} fp4_status;

typedef enum { FP4_NVFP4 = 0, FP4_MXFP4 = 1 } fp4_format;

/* FP4_SCALE_DYNAMIC: the activation global scale is amax / 2688 over the whole
 * tensor, computed on the device per call.  FP4_SCALE_STATIC: the caller
 * supplies it (a checkpoint's input_scale); there is no default, so a missing
 * scale is an error and never a silent zero ("GLM-5.3-Flash on vLLM, on
 * GB10": a weight-only checkpoint left the MoE activation scale at zero).
 * MXFP4 has no global scale and accepts FP4_SCALE_DYNAMIC only. */
typedef enum { FP4_SCALE_DYNAMIC = 0, FP4_SCALE_STATIC = 1 } fp4_scale_mode;

/* ------------------------------------------------------------ utilities */

int fp4_abi_version(void);
const char* fp4_status_string(int status);
/* Message of the last failing call on this host thread ("" if none). */
const char* fp4_last_error_message(void);

/* Byte sizes of the quantised representation of a [rows, k] tensor. */
size_t fp4_codes_bytes(int64_t rows, int64_t k);
size_t fp4_scales_bytes(int fmt, int64_t rows, int64_t k);

/* Synchronises `stream`, then reports and clears the device-side error flags
 * (FP4_ERR_DEVICE_TIMEOUT if any bounded wait gave up since the last call). */
fp4_status fp4_device_status(void* stream);

/* Test hook: pretend the current device has compute capability `sm` (e.g. 90)
 * for the architecture check; 0 restores the real query.  Host-side only. */
void fp4_set_arch_override(int sm);

/* Tuning and test hook (no counterpart on the pages): which kernels fp4_gemm /
 * fp4_gemm_prequant use.  0 = automatic: for m > 64 the one-CTA kernel
 * (128- or 256-wide tiles); for fp4_gemm with m <= 8, k <= 8192 and
 * n >= 64 x (SM count) the fused decode kernel (activation quantisation inside
 * the GEMM launch, one CTA per 128 weight rows); otherwise for m <= 64 the
 * quantiser and a swapped-operand GEMM, split along K (with a reduction
 * launch) when n has fewer than 64 x (SM count) rows.
 * 1 = the one-CTA kernel and never the fused decode kernel; 2 = the CTA-pair
 * kernel (tcgen05 cta_group::2, 256 x 256 tiles) wherever m >= 256 and
 * n >= 256; 3 = the fused decode kernel for every fp4_gemm with m <= 8 and
 * k <= 8192; 4 = fp4_gemm_w4a16 always on its tensor-core kernel (policy 0
 * takes it for m >= 3 when the weight's 128-row tiles fill at least half the
 * SMs, else the CUDA-core kernel); 5 = for m > 64 with 256-wide tiles, an
 * even number of 128-row activation tiles and a pair unit for every cluster,
 * the one-CTA kernel in clusters of two CTAs whose two activation tiles share
 * each 256-row weight tile (each CTA multicasts one half of it into both).
 * Process-wide, host-side; results agree within the GEMM tolerance under every
 * policy (codes and scales are identical).
 * FP4_ERR_INVALID_ARG for a value outside 0..5 (the policy is unchanged). */
fp4_status fp4_set_gemm_tile_policy(int policy);

/* Tuning and test hook (no counterpart on the pages): which implementation
 * fp4_moe_grouped uses.  The one-launch MoE (a memset of its counters, then
 * one cooperative kernel: route, quantise, GEMM1 + SwiGLU, requantise, GEMM2
 * and the top-k sum in slot order) takes 1 <= T <= 16 tokens, top_k <= 8,
 * n_experts <= 256, hidden and inter multiples of 256 and at most 2048;
 * otherwise the launch chain runs.  0 = automatic: the one launch wherever
 * it applies (it is the faster there), else the chain; 1 = always the
 * chain; 2 = the one launch wherever it applies.  Results agree within the MoE tolerance under all.
 * Process-wide, host-side; FP4_ERR_INVALID_ARG for a value outside 0..2. */
fp4_status fp4_set_moe_policy(int policy);

/* Test hook (host-side, no device needed): the plan fp4_gemm /
 * fp4_gemm_prequant would use for an m x n x k GEMM on a device with
 * `sm_count` SMs under the current tile policy.  out[0] = 1 for the
 * small-m (swapped-operand) path, out[1] = the tile width on the MMA's N side,
 * out[2] = the number of K splits, out[3] = 1 for the CTA-pair kernel,
 * out[4] = 1 when fp4_gemm takes the fused decode kernel, and (max_out >= 6)
 * out[5] = 1 for the weight-tile-sharing CTA pairs.  max_out >= 5. */
fp4_status fp4_debug_plan_gemm(int64_t m, int64_t n, int64_t k, int sm_count, int64_t* out, int max_out);

/* Test hook for failure detection: launches one tiny kernel whose thread waits
 * on a barrier that nothing completes, with a wait limit of `limit_us`
 * microseconds; the wait gives up, sets the device flag and returns, leaving
 * the context usable.  Follow with fp4_device_status(). */
fp4_status fp4_debug_timeout_probe(int64_t limit_us, void* stream);

/* ------------------------------------------------- activation quantiser */

size_t fp4_quantize_workspace_size(int fmt, int64_t rows, int64_t k);

/*
 * Quantise a bf16 tensor x [rows, k] to `fmt`.
 * NVFP4 ("vLLM on DGX Spark: technical report", section 6.1): per 16-element
 * block amax_b, block scale s_b = E4M3_rne_satfinite(amax_b / (6 s_g)),
 * d = s_b s_g, element = E2M1_rne_satfinite(x / d) (0 when d is 0); s_g is
 * amax / 2688 (dynamic) or static_scale (static).  s_g is written to
 * *global_scale (device fp32).
 * MXFP4 (same page, section 6.4): per 32-element block, E8M0 exponent
 * floor(log2 amax_b) - 2, element = E2M1_rne_satfinite(x / 2^e); all-zero
 * blocks get byte 0; *global_scale (if not NULL) is set to 1.
 * Outputs: codes (fp4_codes_bytes), scales in the MMA layout
 * (fp4_scales_bytes, padding zeroed).  Bit-exact with the CPU oracle.
 */
fp4_status fp4_quantize_act(int fmt, const void* x_bf16, int64_t rows, int64_t k, int mode, float static_scale,
                            void* codes, void* scales, float* global_scale, void* workspace, size_t workspace_bytes,
                            void* stream);

/* fp4_quantize_act without a workspace, for callers that cannot allocate
 * device memory: code that runs under another component's memory plan (a
 * framework that forbids allocation on its hot path, a pre-built CUDA graph
 * with fixed buffers, a real-time loop) or a C caller with no device
 * allocator.  No layer the source pages describe has this entry point.
 * Same arguments, results and errors as fp4_quantize_act, minus the
 * workspace: the dynamic NVFP4 amax partials go to a static device array of
 * 1024 floats (4 KiB) that every GPU loading the library keeps until the
 * process exits; a launch that would need more partial slots is rejected with
 * FP4_ERR_WORKSPACE.  No cudaMalloc / cudaFree or allocating library call is
 * made.  The first call on each device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the array, so calls that
 * overlap on the GPU (other streams, other host threads) race; the array keeps
 * the last call's contents, and every slot a call reads is written earlier
 * in that same call. */
fp4_status fp4_quantize_act_noalloc(int fmt, const void* x_bf16, int64_t rows, int64_t k, int mode,
                                    float static_scale, void* codes, void* scales, float* global_scale,
                                    void* stream);

/* Weight preparation (done once at load time, not on the hot path): the same
 * quantiser with a dynamic per-tensor scale, w [n, k] -> codes, MMA-layout
 * scales and *global_scale.  The scale layout conversion to the MMA layout
 * happens here, once ("vLLM on DGX Spark: technical report", section 4.3:
 * scale factors are converted to the MMA layout once after loading). */
fp4_status fp4_prepack_weight(int fmt, const void* w_bf16, int64_t n, int64_t k, void* codes, void* scales,
                              float* global_scale, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------- linear layer */

size_t fp4_gemm_workspace_size(int fmt, int64_t m, int64_t n, int64_t k);

/*
 * W4A4 linear: out[m, n] = bf16( alpha * sum_k deq(A)[m, k] * deq(W)[n, k] ),
 * alpha = s_gA * s_gW in fp32 (MXFP4: 1), fp32 accumulation on the tensor
 * cores ("vLLM on DGX Spark: technical report", sections 6.1-6.3).
 * x_bf16 [m, k] is quantised on the device per call (mode / static_scale as
 * in fp4_quantize_act; NVFP4 only for static); the weight is pre-quantised
 * (fp4_prepack_weight): w_codes [n, k/2], w_scales MMA layout, w_global one
 * device fp32 (ignored for MXFP4, may be NULL).  out_bf16 [m, n] row-major.
 * Small m (decode) runs a weight-streaming variant with the same numerics.
 * workspace: fp4_gemm_workspace_size(fmt, m, n, k) bytes, 256-byte aligned.
 */
fp4_status fp4_gemm(int fmt, const void* x_bf16, int64_t m, int mode, float static_scale, const void* w_codes,
                    const void* w_scales, const float* w_global, int64_t n, int64_t k, void* out_bf16,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Same GEMM with A already quantised (a_codes [m, k/2], a_scales MMA layout,
 * a_global one device fp32, ignored for MXFP4).  workspace may be NULL when
 * fp4_gemm_prequant_workspace_size() is 0. */
size_t fp4_gemm_prequant_workspace_size(int fmt, int64_t m, int64_t n, int64_t k);
fp4_status fp4_gemm_prequant(int fmt, const void* a_codes, const void* a_scales, const float* a_global, int64_t m,
                             const void* w_codes, const void* w_scales, const float* w_global, int64_t n, int64_t k,
                             void* out_bf16, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------- MXFP8 / MXFP6 (8-bit containers) */

/* Element formats of the wider MX formats ("vLLM per-format kernel capability
 * matrix": MXFP6 and MXFP8 with group size 32): MXFP8 with E4M3 or E5M2
 * elements, MXFP6 with E2M3 or E3M2 elements. */
typedef enum { FP4_MX_E4M3 = 0, FP4_MX_E5M2 = 1, FP4_MX_E2M3 = 2, FP4_MX_E3M2 = 3 } fp4_mx_elem;

/*
 * MX quantiser with 8-bit containers.  Per 32-element block of a row,
 * e = floor(log2 amax_b) - emax (emax = the element's largest exponent: E4M3
 * 8, E5M2 15, E2M3 2, E3M2 4), clamped to [-127, 127], stored as the E8M0
 * byte e + 127 -- the MXFP4 rule of "vLLM on DGX Spark: technical report",
 * section 6.4, with the element's own emax; each element is
 * ELEM_rne_satfinite(x * 2^-e) (saturating at the largest finite value:
 * 448, 57344, 7.5, 28; the sign of a value that rounds to zero kept); an
 * all-zero block gets scale byte 0 and code 0.
 * x_bf16 [rows, k]; codes [rows, k], ONE BYTE PER ELEMENT (the FP6 codes in
 * the low six bits, the top two bits 0: the layout the tensor cores read from
 * shared memory, so MXFP6 is not packed to 6 bits in memory); scales in the
 * MMA layout of MXFP4 (fp4_scales_bytes(FP4_MXFP4, rows, k) bytes, padding
 * written as 0).  All 16-byte aligned; k a positive multiple of 32.  No
 * workspace.  FP4_ERR_INVALID_ARG for an unknown element format.
 */
fp4_status fp4_quantize_mx(int elem, const void* x_bf16, int64_t rows, int64_t k, void* codes, void* scales,
                           void* stream);

/* fp4_quantize_mx with E4M3 elements (MXFP8). */
fp4_status fp4_quantize_mxfp8(const void* x_bf16, int64_t rows, int64_t k, void* codes, void* scales, void* stream);

/*
 * MXFP6 codes (E2M3 or E3M2, one per byte as fp4_quantize_mx writes them) ->
 * the E4M3 codes of the same values, [rows, k] bytes; out may equal codes
 * (in place).  Every E2M3 and E3M2 value is an E4M3 value, so this is exact
 * and the E8M0 scales stay as they are: an MXFP6 operand widened this way
 * (weights once at load) goes through the MX GEMM as FP4_MX_E4M3 and the
 * products are those of the MXFP6 values.  FP4_ERR_INVALID_ARG for an MXFP8
 * element format.
 */
fp4_status fp4_mx_widen(int elem, const void* codes, int64_t rows, int64_t k, void* out, void* stream);

/*
 * MX linear (MXFP8 operands, E4M3 or E5M2 elements, either on either side):
 * out[m, n] = bf16( sum_k deq(A)[m, k] * deq(W)[n, k] ) with deq = element x
 * 2^(scale byte - 127) per 32-element block, fp32 accumulation on the tensor
 * cores (tcgen05 kind::mxf8f6f4); no global scale.  a_codes [m, k] /
 * w_codes [n, k] and their scales as written by fp4_quantize_mx (a_elem /
 * w_elem name their element formats: FP4_MX_E4M3 or FP4_MX_E5M2; MXFP6
 * operands are passed widened by fp4_mx_widen as FP4_MX_E4M3, and an
 * unwidened MXFP6 format gives FP4_ERR_INVALID_ARG).
 * out_bf16 [m, n] row-major.  k a multiple of 32 (16-byte code rows), n a
 * multiple of 8.  No workspace.
 */
fp4_status fp4_gemm_mx_prequant(int a_elem, const void* a_codes, const void* a_scales, int64_t m, int w_elem,
                                const void* w_codes, const void* w_scales, int64_t n, int64_t k, void* out_bf16,
                                void* stream);

/* The same linear with the bf16 activations x_bf16 [m, k] quantised to a_elem
 * on the device per call (fp4_quantize_mx into the workspace, then the GEMM);
 * a_elem may be an MXFP6 format here (the codes are widened as they are
 * written), w_elem is E4M3 or E5M2 (MXFP6 weights widened at load).
 * workspace: fp4_gemm_mx_workspace_size(m, k) bytes, 256-byte aligned. */
size_t fp4_gemm_mx_workspace_size(int64_t m, int64_t k);
fp4_status fp4_gemm_mx(int a_elem, const void* x_bf16, int64_t m, int w_elem, const void* w_codes,
                       const void* w_scales, int64_t n, int64_t k, void* out_bf16, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Weight-only (W4A16) linear for decode: out[m, n] = bf16( s_gW * sum_k
 * x[m, k] * E2M1(w)[n, k] * s_b[n, k / B] ) with the bf16 activations used as
 * they are, not quantised ("vLLM on DGX Spark: technical report", section 5.3
 * "Marlin for NVFP4": the FP4 weight is dequantised to 16 bits and multiplied
 * with 16-bit activations).  B = 16 (NVFP4, s_gW = *w_global) or 32 (MXFP4,
 * s_gW = 1, w_global ignored and may be NULL).  Each product of an element and
 * its block scale is exact in fp32; the sum is fp32 in an unspecified order,
 * then one bf16 rounding.  The weight is the prepacked one of fp4_gemm.
 * x_bf16 [m, k], out_bf16 [m, n] row-major, 16-byte aligned.  Requires
 * m <= 4 and k <= 8192 (FP4_ERR_SHAPE otherwise); no workspace; one launch
 * that reads every weight byte once.
 */
fp4_status fp4_gemm_w4a16(int fmt, const void* x_bf16, int64_t m, const void* w_codes, const void* w_scales,
                          const float* w_global, int64_t n, int64_t k, void* out_bf16, void* stream);

/* ---------------------------------------------------------- fused MoE */

/*
 * NVFP4 expert weights, prepared once: w13 [E, 2I, H] bf16 (rows 0..I-1 gate,
 * rows I..2I-1 up), w2 [E, H, I] bf16.  Each expert is quantised with its own
 * dynamic global scale (w13_global[e], w2_global[e], device fp32 [E]).  The
 * w13 rows are stored interleaved in groups of 32 (gate 0-31, up 0-31, gate
 * 32-63, up 32-63, ...) so that a GEMM tile holds matching gate and up rows;
 * w13_codes [E*2I, H/2], w13_scales = fp4_scales_bytes(NVFP4, E*2I, H);
 * w2_codes [E*H, I/2], w2_scales = fp4_scales_bytes(NVFP4, E*H, I).
 * Requires I % 64 == 0 and H % 128 == 0.
 */
size_t fp4_moe_prepack_workspace_size(int64_t n_experts, int64_t hidden, int64_t inter);
fp4_status fp4_moe_prepack_weights(const void* w13_bf16, const void* w2_bf16, int64_t n_experts, int64_t hidden,
                                   int64_t inter, void* w13_codes, void* w13_scales, float* w13_global,
                                   void* w2_codes, void* w2_scales, float* w2_global, void* workspace,
                                   size_t workspace_bytes, void* stream);

size_t fp4_moe_workspace_size(int64_t tokens, int64_t hidden, int64_t inter, int64_t n_experts, int64_t top_k);

/*
 * Fused MoE forward, the stages of "vLLM on DGX Spark: technical report",
 * section 7.1 (router -> quantise/dispatch -> permute, experts, unpermute ->
 * combine) with the expert computation of section 4.3 (two GEMMs, SwiGLU,
 * top-k weighted reduction):
 *   1. router: p = softmax(logits[t]); top_k experts by p (ties: lower index);
 *      weights renormalised over the top_k.
 *   2. permute: assignments sorted by (expert, token, slot).
 *   3. hidden [T, H] quantised to NVFP4 once (dynamic per-tensor s_gA; static:
 *      per-expert static_scales13[e] for that expert's rows).
 *   4. per expert e: G = alpha1_e * A_q . W13_e^T (alpha1_e = s_gA * w13_global[e]),
 *      h = bf16(SiLU(G_gate) * G_up), and the per-expert amax of h.
 *   5. h requantised to NVFP4 with s_gH[e] = amax_e / 2688 (static:
 *      static_scales2[e]).
 *   6. D = alpha2_e * H_q . W2_e^T (alpha2_e = s_gH[e] * w2_global[e]).
 *   7. out[t] = bf16( sum_j weight[t, j] * D[t, j] ): D kept in fp32 (one row
 *      per routing slot, in the expert-sorted row order), the top_k terms
 *      added in fp32 in slot order j = 0..top_k-1, so the result is the same
 *      bits on every run.
 * hidden_bf16 [T, H], router_logits fp32 [T, E], out_bf16 [T, H] (device).
 * mode FP4_SCALE_STATIC needs both host arrays static_scales13[E] and
 * static_scales2[E] (each finite and > 0, E <= 256): NULL gives
 * FP4_ERR_MISSING_SCALE, a zero / negative / NaN scale FP4_ERR_INVALID_SCALE.
 * A weight-only checkpoint passes FP4_SCALE_DYNAMIC.  top_k <= n_experts <= 1024.
 * workspace: fp4_moe_workspace_size(...) bytes.
 */
fp4_status fp4_moe_grouped(const void* hidden_bf16, const float* router_logits, int64_t tokens, int64_t hidden,
                           int64_t inter, int64_t n_experts, int64_t top_k, int mode, const float* static_scales13,
                           const float* static_scales2, const void* w13_codes, const void* w13_scales,
                           const float* w13_global, const void* w2_codes, const void* w2_scales,
                           const float* w2_global, void* out_bf16, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Staged variant for stage-by-stage checks: runs only the stages whose bit is
 * set in stage_mask (bit 0 router+permute, 1 quantise/dispatch hidden, 2
 * GEMM1+SiLU*up, 3 requantise h, 4 GEMM2+combine) and leaves every
 * intermediate in the workspace at the byte offsets reported by
 * fp4_moe_workspace_layout(); a stage reads its inputs from there, so a
 * caller may place its own values before running a later stage.  Offsets[]:
 * 0 ids int32 [T*k], 1 weights fp32 [T*k], 2 expert offsets int32 [E+1]
 * (unpadded), 3 padded row offsets int32 [E+1], 4 source slot of each padded
 * row int32 [R] (-1 for padding), 5 A codes [R, H/2], 6 A scales (MMA layout,
 * R rows), 7 s_gA / static scale per expert fp32 [E], 8 h bf16 [R, I],
 * 9 amax of h per expert fp32 [E], 10 s_gH fp32 [E], 11 h codes [R, I/2],
 * 12 h scales (MMA layout), 13 D = alpha2 x GEMM2, fp32 [R, H], one row per
 * padded row (the row of slot t * top_k + j is the one entry 4 maps to it); R = offsets
 * count 14 (the padded row capacity).  Entries 15-21 are written by the
 * one-launch MoE (regions sized only for the shapes it takes), all in slot
 * order t * top_k + j: 15 h bf16 [T*k, I], 16 the requantised h codes
 * [T*k, I/2], 17 their scale bytes [T*k, I/16] (row-major, not the MMA
 * layout), 18 s_gH fp32 [E] (the experts with tokens), 19 D = alpha2 x GEMM2
 * fp32 [T*k, H], 20 the dispatched hidden codes [T*k, H/2], 21 their scale
 * bytes [T*k, H/16]; that form also writes entries 0 and 1 and (dynamic
 * scale) s_gA in entry 7.  Returns the number of entries written. */
int fp4_moe_workspace_layout(int64_t tokens, int64_t hidden, int64_t inter, int64_t n_experts, int64_t top_k,
                             int64_t* offsets, int max_entries);
fp4_status fp4_moe_grouped_stages(const void* hidden_bf16, const float* router_logits, int64_t tokens,
                                  int64_t hidden, int64_t inter, int64_t n_experts, int64_t top_k, int mode,
                                  const float* static_scales13, const float* static_scales2, const void* w13_codes,
                                  const void* w13_scales, const float* w13_global, const void* w2_codes,
                                  const void* w2_scales, const float* w2_global, void* out_bf16, void* workspace,
                                  size_t workspace_bytes, unsigned stage_mask, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4_H */
