/*
 * fp4_oracle.c -- plain, slow CPU oracle for block-scaled FP4 (NVFP4 / MXFP4).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no FMA contraction, IEEE single precision for every float operation, so the
 * arithmetic below is exactly the fp32 sequence written in the source).
 *
 * Sources (page title, section):
 *  - "vLLM on DGX Spark: technical report", section 6.1 "NVFP4 format":
 *    E2M1 elements (2-bit exponent, 1-bit mantissa, max 6.0) packed two per
 *    byte, one FP8-E4M3 scale per 16 contiguous elements along K, one fp32
 *    global scale per tensor; value = element x block scale x global scale.
 *  - same page, section 6.4 "NVFP4 vs MXFP4": MXFP4 has 32-element K blocks
 *    and exponent-only E8M0 scales.
 *  - the E2M1 value set {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6} and the
 *    dynamic global scale amax / (6 * 448) are the workload's own definitions.
 *
 * Readings where the pages are silent are listed at each function.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ bf16 */

/* bf16 is the upper half of an IEEE binary32. */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even fp32 -> bf16 (finite inputs; NaN kept quiet). */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------ E2M1 */

/* Magnitudes of the eight non-negative E2M1 codes, by code index 0..7. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float orc_e2m1_decode(uint8_t code) {
    double m = E2M1_MAG[code & 7u];
    return (float)((code & 8u) ? -m : m);
}

/*
 * Nearest grid point, ties to the code whose mantissa bit (= code bit 0) is 0,
 * magnitudes above 6 saturate to 6 (satfinite).  Reading where the pages are
 * silent: the sign bit is kept, so a negative value that rounds to zero gives
 * code 0x8 (negative zero).
 */
uint8_t orc_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 8u : 0u;
    double a = fabs((double)v);
    if (a >= 6.0) return (uint8_t)(sign | 7u);
    int lo = 0;
    while (lo < 7 && E2M1_MAG[lo + 1] <= a) lo++;
    if (E2M1_MAG[lo] == a) return (uint8_t)(sign | (uint8_t)lo);
    double dlo = a - E2M1_MAG[lo];
    double dhi = E2M1_MAG[lo + 1] - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = lo + 1;
    else c = (lo & 1) ? lo + 1 : lo;
    return (uint8_t)(sign | (uint8_t)c);
}

/* ------------------------------------------------------------------ E4M3 */

/* OCP FP8 E4M3 ("fn"): bias 7, no infinities, 0x7F / 0xFF are NaN, max 448. */
static double e4m3_mag(int b7) {
    int e = (b7 >> 3) & 0xF, m = b7 & 7;
    if (e == 0) return ldexp((double)m, -9);
    return ldexp((double)(8 + m), e - 10);
}

float orc_e4m3_decode(uint8_t b) {
    if ((b & 0x7Fu) == 0x7Fu) return NAN;
    double m = e4m3_mag(b & 0x7F);
    return (float)((b & 0x80u) ? -m : m);
}

/* Round to nearest even on the E4M3 grid; magnitudes >= 448 (and +inf) give
 * 448 (satfinite).  NaN input is outside the contract and returns 0x7F. */
uint8_t orc_e4m3_encode(float v) {
    if (isnan(v)) return 0x7Fu;
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    int lo = 0;
    while (lo < 0x7E && e4m3_mag(lo + 1) <= a) lo++;
    if (e4m3_mag(lo) == a) return (uint8_t)(sign | (uint8_t)lo);
    double dlo = a - e4m3_mag(lo);
    double dhi = e4m3_mag(lo + 1) - a;
    int c;
    if (dlo < dhi) c = lo;
    else if (dhi < dlo) c = lo + 1;
    else c = (lo & 1) ? lo + 1 : lo;
    return (uint8_t)(sign | (uint8_t)c);
}

/* ------------------------------------------------------------------ E8M0 */

/* Exponent-only scale: 2^(b - 127); 0xFF is NaN. */
float orc_e8m0_decode(uint8_t b) {
    if (b == 0xFFu) return NAN;
    return ldexpf(1.0f, (int)b - 127);
}

/* ------------------------------------------------------ scale MMA layout */

/*
 * Block scales are kept two ways: canonical [rows][ksf] (one byte per K block,
 * row-major) and the "MMA layout" the tensor cores read, which the GPU path
 * uses in memory.  Rows are padded to a multiple of 128 and the scale columns
 * to whole 256-element K tiles (16 NVFP4 / 8 MXFP4 scale columns); padding
 * bytes are 0.  The layout groups 128 rows x 4 scale columns into one 512-byte
 * atom; inside an atom, row r sits at byte (r % 32) * 16 + (r / 32) * 4 and
 * scale column j at + (j % 4).  Atoms are ordered row-tile major, then K.
 */
int64_t orc_scale_cols_padded(int64_t k, int64_t block) {
    int64_t k_pad = (k + 255) / 256 * 256;
    return k_pad / block;
}

int64_t orc_scale_mma_bytes(int64_t rows, int64_t k, int64_t block) {
    int64_t rows_pad = (rows + 127) / 128 * 128;
    return rows_pad * orc_scale_cols_padded(k, block);
}

int64_t orc_scale_mma_index(int64_t row, int64_t j, int64_t ksf_pad) {
    int64_t atoms_per_rowtile = ksf_pad / 4;
    int64_t atom = (row / 128) * atoms_per_rowtile + j / 4;
    int64_t r = row % 128;
    return atom * 512 + (r % 32) * 16 + (r / 32) * 4 + (j % 4);
}

/* canonical [rows][ksf] -> MMA layout (zero-filled padding). */
void orc_scales_to_mma(const uint8_t* canon, int64_t rows, int64_t k, int64_t block, uint8_t* mma) {
    int64_t ksf = k / block;
    int64_t ksf_pad = orc_scale_cols_padded(k, block);
    memset(mma, 0, (size_t)orc_scale_mma_bytes(rows, k, block));
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < ksf; j++) mma[orc_scale_mma_index(r, j, ksf_pad)] = canon[r * ksf + j];
}

/* MMA layout -> canonical [rows][ksf]. */
void orc_scales_from_mma(const uint8_t* mma, int64_t rows, int64_t k, int64_t block, uint8_t* canon) {
    int64_t ksf = k / block;
    int64_t ksf_pad = orc_scale_cols_padded(k, block);
    for (int64_t r = 0; r < rows; r++)
        for (int64_t j = 0; j < ksf; j++) canon[r * ksf + j] = mma[orc_scale_mma_index(r, j, ksf_pad)];
}

/* ------------------------------------------------------------ amax */

/* Exact max |x| over n bf16 values (max is exact in any precision). */
float orc_amax_bf16(const uint16_t* x, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(orc_bf16_to_f32(x[i]));
        if (a > m) m = a;
    }
    return m;
}

/* Dynamic per-tensor global scale (dequant convention): amax / (6 * 448). */
float orc_nvfp4_global_scale(float amax) { return amax / 2688.0f; }

/* --------------------------------------------------------- NVFP4 quantise */

/*
 * Quantise rows x k bf16 values with a given fp32 global scale s_g (dequant
 * convention: value ~= code * block_scale * s_g).  For each 16-element block:
 *   amax_b = max |x|,   p = fl(s_g * 6),   t = fl(amax_b / p),
 *   s_b    = E4M3_rne_satfinite(t)           (0 when p is 0),
 *   d      = fl(decode(s_b) * s_g),
 *   q_i    = E2M1_rne_satfinite(fl(x_i / d)) (all 0 when d is 0).
 * Readings: correctly rounded division (not a reciprocal multiply), scales
 * rounded to nearest even, saturation instead of rescaling.
 * Packing: element 2j in the low nibble of byte j of the row.
 * codes: [rows][k/2], scales: canonical [rows][k/16].
 */
void orc_quantize_nvfp4_given_scale(const uint16_t* x, int64_t rows, int64_t k, float s_g, uint8_t* codes,
                                    uint8_t* scales) {
    int64_t nb = k / 16;
    float p = s_g * 6.0f;
    for (int64_t r = 0; r < rows; r++) {
        const uint16_t* xr = x + r * k;
        for (int64_t b = 0; b < nb; b++) {
            float xv[16];
            float amax_b = 0.0f;
            for (int i = 0; i < 16; i++) {
                xv[i] = orc_bf16_to_f32(xr[b * 16 + i]);
                float a = fabsf(xv[i]);
                if (a > amax_b) amax_b = a;
            }
            uint8_t sb = 0;
            if (p > 0.0f) {
                float t = amax_b / p;
                sb = orc_e4m3_encode(t);
            }
            float d = orc_e4m3_decode(sb) * s_g;
            scales[r * nb + b] = sb;
            for (int i = 0; i < 16; i += 2) {
                uint8_t lo = 0, hi = 0;
                if (d != 0.0f) {
                    lo = orc_e2m1_encode(xv[i] / d);
                    hi = orc_e2m1_encode(xv[i + 1] / d);
                }
                codes[r * (k / 2) + (b * 16 + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/*
 * Per-tensor NVFP4 quantisation.  mode 0 = dynamic: s_g = amax / 2688 over the
 * whole tensor.  mode 1 = static: s_g = static_scale (the checkpoint's
 * activation scale, dequant convention).  Returns s_g through *s_g_out.
 */
void orc_quantize_nvfp4(const uint16_t* x, int64_t rows, int64_t k, int mode, float static_scale, uint8_t* codes,
                        uint8_t* scales, float* s_g_out) {
    float s_g = (mode == 0) ? orc_nvfp4_global_scale(orc_amax_bf16(x, rows * k)) : static_scale;
    orc_quantize_nvfp4_given_scale(x, rows, k, s_g, codes, scales);
    *s_g_out = s_g;
}

/* --------------------------------------------------------- MXFP4 quantise */

/*
 * MXFP4: per 32-element block, shared exponent e = floor(log2(amax_b)) - 2
 * (2 = the largest E2M1 exponent), clamped to [-127, 127], stored as the
 * E8M0 byte e + 127; q_i = E2M1_rne_satfinite(x_i / 2^e) (exact division).
 * Reading where the pages are silent: an all-zero block gets scale byte 0x00
 * and zero codes; values in (6, 8) * 2^e saturate to 6.
 * codes: [rows][k/2], scales: canonical [rows][k/32].
 */
void orc_quantize_mxfp4(const uint16_t* x, int64_t rows, int64_t k, uint8_t* codes, uint8_t* scales) {
    int64_t nb = k / 32;
    for (int64_t r = 0; r < rows; r++) {
        const uint16_t* xr = x + r * k;
        for (int64_t b = 0; b < nb; b++) {
            float xv[32];
            float amax_b = 0.0f;
            for (int i = 0; i < 32; i++) {
                xv[i] = orc_bf16_to_f32(xr[b * 32 + i]);
                float a = fabsf(xv[i]);
                if (a > amax_b) amax_b = a;
            }
            if (amax_b == 0.0f) {
                scales[r * nb + b] = 0;
                for (int i = 0; i < 32; i += 2) codes[r * (k / 2) + (b * 32 + i) / 2] = 0;
                continue;
            }
            int ex;
            frexpf(amax_b, &ex); /* amax_b = f * 2^ex, f in [0.5, 1) */
            int e = (ex - 1) - 2;
            if (e < -127) e = -127;
            if (e > 127) e = 127;
            scales[r * nb + b] = (uint8_t)(e + 127);
            float X = ldexpf(1.0f, e);
            for (int i = 0; i < 32; i += 2) {
                uint8_t lo = orc_e2m1_encode(xv[i] / X);
                uint8_t hi = orc_e2m1_encode(xv[i + 1] / X);
                codes[r * (k / 2) + (b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* ------------------------------------------------------------ dequantise */

/* fmt 0 = NVFP4 (block 16, E4M3 scales, global scale s_g),
 * fmt 1 = MXFP4 (block 32, E8M0 scales, no global scale: s_g ignored).
 * Writes rows x k doubles: code x block scale (x s_g for NVFP4 when
 * apply_global != 0). */
void orc_dequantize(int fmt, const uint8_t* codes, const uint8_t* scales, float s_g, int apply_global, int64_t rows,
                    int64_t k, double* out) {
    int64_t block = fmt == 0 ? 16 : 32;
    int64_t nb = k / block;
    for (int64_t r = 0; r < rows; r++)
        for (int64_t i = 0; i < k; i++) {
            uint8_t byte = codes[r * (k / 2) + i / 2];
            uint8_t c = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
            uint8_t sb = scales[r * nb + i / block];
            double s = fmt == 0 ? (double)orc_e4m3_decode(sb) : (double)orc_e8m0_decode(sb);
            double v = (double)orc_e2m1_decode(c) * s;
            if (fmt == 0 && apply_global) v *= (double)s_g;
            out[r * k + i] = v;
        }
}

/* ------------------------------------------------------- exact NVFP4 GEMM */

/*
 * S[m][n] = sum_k deqA[m][k] * deqB[n][k] without the global scales, exactly:
 * 2*E2M1 is an integer in [-12, 12] and 2^9*E4M3 an integer below 2^18, so
 * each product scaled by 2^20 is an integer below 2^43 and the K-sum fits in
 * int64 for K < 2^20.  Returns S * 2^20 as int64 (row-major [m][n]).  Scales
 * are canonical [rows][k/16].  Used as an independent check on the
 * dequantise-then-fp64 GEMM.
 */
void orc_gemm_nvfp4_exact(const uint8_t* ca, const uint8_t* sa, const uint8_t* cb, const uint8_t* sb, int64_t M,
                          int64_t N, int64_t K, int64_t* S20) {
    int64_t nb = K / 16;
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            int64_t acc = 0;
            for (int64_t i = 0; i < K; i++) {
                uint8_t ba = ca[m * (K / 2) + i / 2], bb = cb[n * (K / 2) + i / 2];
                uint8_t qa = (i & 1) ? (uint8_t)(ba >> 4) : (uint8_t)(ba & 15u);
                uint8_t qb = (i & 1) ? (uint8_t)(bb >> 4) : (uint8_t)(bb & 15u);
                int64_t ea = (int64_t)llround(2.0 * (double)orc_e2m1_decode(qa));
                int64_t eb = (int64_t)llround(2.0 * (double)orc_e2m1_decode(qb));
                int64_t fa = (int64_t)llround(512.0 * (double)orc_e4m3_decode(sa[m * nb + i / 16]));
                int64_t fb = (int64_t)llround(512.0 * (double)orc_e4m3_decode(sb[n * nb + i / 16]));
                acc += ea * eb * fa * fb;
            }
            S20[m * N + n] = acc;
        }
}
