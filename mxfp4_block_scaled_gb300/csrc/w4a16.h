// w4a16.h -- launcher of the weight-only FP4 linear (w4a16.cu), for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fp4 {

constexpr int kW4A16MaxM = 4;     // activation rows of fp4_gemm_w4a16
constexpr int kW4A16MaxK = 8192;  // the activations are staged in shared memory

// out [m][n] bf16 = bf16(s_gW * x [m][k] . dequant(W [n][k])^T); fmt as in fp4.h.
cudaError_t launch_w4a16(int fmt, const uint16_t* x, int m, int64_t n, int64_t k, const uint8_t* w_codes,
                         const uint8_t* w_scales, const float* w_global, uint16_t* out, cudaStream_t s);

// The same on the tensor cores (w4a16_tc.cu): one CTA per 128 weight rows,
// the weights dequantised to bf16 in shared memory, kind::f16 MMAs (m <= 16).
cudaError_t launch_w4a16_tc(int fmt, const uint16_t* x, int m, int64_t n, int64_t k, const uint8_t* w_codes,
                            const uint8_t* w_scales, const float* w_global, uint16_t* out, cudaStream_t s);

}  // namespace fp4
