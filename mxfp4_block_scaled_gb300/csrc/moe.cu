// moe.cu -- fused-MoE pipeline (entry points stubbed until the kernels land).
#include "common.cuh"
#include "internal.h"

using namespace fp4;

extern "C" size_t fp4_moe_prepack_workspace_size(int64_t, int64_t, int64_t) { return 4096; }
extern "C" fp4_status fp4_moe_prepack_weights(const void*, const void*, int64_t, int64_t, int64_t, void*, void*, float*,
                                              void*, void*, float*, void*, size_t, void*) {
    set_error("MoE not built yet");
    return FP4_ERR_INVALID_ARG;
}
extern "C" size_t fp4_moe_workspace_size(int64_t, int64_t, int64_t, int64_t, int64_t) { return 0; }
extern "C" int fp4_moe_workspace_layout(int64_t, int64_t, int64_t, int64_t, int64_t, int64_t*, int) { return 0; }
extern "C" fp4_status fp4_moe_grouped(const void*, const float*, int64_t, int64_t, int64_t, int64_t, int64_t, int,
                                      const float*, const float*, const void*, const void*, const float*,
                                      const void*, const void*, const float*, void*, void*, size_t, void*) {
    set_error("MoE not built yet");
    return FP4_ERR_INVALID_ARG;
}
extern "C" fp4_status fp4_moe_grouped_stages(const void*, const float*, int64_t, int64_t, int64_t, int64_t, int64_t,
                                             int, const float*, const float*, const void*, const void*,
                                             const float*, const void*, const void*, const float*, void*, void*,
                                             size_t, unsigned, void*) {
    set_error("MoE not built yet");
    return FP4_ERR_INVALID_ARG;
}
