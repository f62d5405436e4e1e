// mxfp8.h -- launcher of the MXFP8 (E4M3) quantiser (mxfp8.cu), for the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fp4 {

// x bf16 [rows][k] -> codes [rows][k] E4M3 bytes, scales E8M0 in the MMA layout.
cudaError_t launch_mxfp8_quant(const uint16_t* x, int64_t rows, int64_t k, uint8_t* codes, uint8_t* scales,
                               int sm_count, cudaStream_t s);

}  // namespace fp4
