// mxfp8.h -- launcher of the MXFP8 / MXFP6 quantisers (mxfp8.cu), for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fp4.h"

namespace fp4 {

// Element formats of the 8-bit-container MX quantisers (the fp4_mx_elem values).
enum : int {
    MX_ELEM_E4M3 = FP4_MX_E4M3,
    MX_ELEM_E5M2 = FP4_MX_E5M2,
    MX_ELEM_E2M3 = FP4_MX_E2M3,
    MX_ELEM_E3M2 = FP4_MX_E3M2,
};

// Exponent of the element format's largest normal value.
__host__ __device__ constexpr int mx_elem_emax(int elem) {
    return elem == MX_ELEM_E4M3 ? 8 : elem == MX_ELEM_E5M2 ? 15 : elem == MX_ELEM_E2M3 ? 2 : 4;
}

// x bf16 [rows][k] -> codes [rows][k], one byte per element, scales E8M0 in
// the MMA layout; with `widen` (E2M3 / E3M2 only) each 6-bit code is written
// as the E4M3 code of the same value.  cudaErrorInvalidValue for an unknown
// element format.
cudaError_t launch_mx8_quant(int elem, const uint16_t* x, int64_t rows, int64_t k, uint8_t* codes, uint8_t* scales,
                             int sm_count, cudaStream_t s, bool widen = false);

// 6-bit codes (E2M3 / E3M2, one per byte) -> the E4M3 codes of the same
// values; bytes % 16 == 0, in may equal out.
cudaError_t launch_mx6_widen(int elem, const uint8_t* in, uint8_t* out, int64_t bytes, int sm_count, cudaStream_t s);

}  // namespace fp4
