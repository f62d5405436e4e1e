// noalloc.cu -- fp4_quantize_act_noalloc: the activation quantiser for
// callers that cannot allocate device memory.
//
// fp4_quantize_act needs a small caller-provided workspace: the dynamic NVFP4
// scale is found by an amax pass that leaves one partial maximum per block
// there for the quantise pass to reduce.  Some callers cannot provide one:
// code running under someone else's memory plan (a framework that forbids
// allocation on its hot path, a pre-built CUDA graph whose buffers are fixed,
// a real-time loop that must not call cudaMalloc) or a plain C caller with no
// device allocator at hand.  This entry point keeps those partials in a
// file-scope device array instead, so the caller passes only the input and
// the three outputs.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4 {

// Scratch for the amax partials: 1024 floats (4 KiB).  Every GPU that loads
// the library holds this array until the process exits.
static constexpr int kNoAllocSlots = 1024;
static __device__ __align__(256) float g_noalloc_partials[kNoAllocSlots];

static std::mutex g_noalloc_mtx;
static float* g_noalloc_ptr[64];  // device address of the array, per device

// Device address of the scratch array for the current device.  The array's
// name is only a host-side stand-in for it, so the address is looked up once
// per device (with that device current) and cached.
static fp4_status noalloc_scratch(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        set_error("no usable CUDA device");
        return FP4_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mtx);
    if (!g_noalloc_ptr[dev]) {
        float* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress((void**)&p, g_noalloc_partials);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            set_error("cudaGetSymbolAddress of the quantiser scratch failed: %s", cudaGetErrorString(e));
            return FP4_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return FP4_OK;
}

}  // namespace fp4

using namespace fp4;

extern "C" fp4_status fp4_quantize_act_noalloc(int fmt, const void* x, int64_t rows, int64_t k, int mode,
                                               float static_scale, void* codes, void* scales, float* global_scale,
                                               void* stream) {
    if (fmt != FP4_NVFP4 && fmt != FP4_MXFP4) {
        set_error("unknown format %d", fmt);
        return FP4_ERR_INVALID_ARG;
    }
    if (rows < 0 || rows >= (1ll << 31)) {
        set_error("rows = %lld out of range", (long long)rows);
        return FP4_ERR_SHAPE;
    }
    if (k <= 0 || k % 32 != 0 || k >= (1ll << 31)) {
        set_error("k = %lld must be a positive multiple of 32", (long long)k);
        return FP4_ERR_SHAPE;
    }
    if (mode != FP4_SCALE_DYNAMIC && mode != FP4_SCALE_STATIC) {
        set_error("unknown scale mode %d", mode);
        return FP4_ERR_INVALID_ARG;
    }
    if (mode == FP4_SCALE_STATIC) {
        if (fmt != FP4_NVFP4) {
            set_error("MXFP4 has no global scale: use FP4_SCALE_DYNAMIC");
            return FP4_ERR_INVALID_ARG;
        }
        if (!(isfinite(static_scale) && static_scale > 0.0f)) {
            set_error("static activation scale %g is not finite and > 0", (double)static_scale);
            return FP4_ERR_INVALID_SCALE;
        }
    }
    if (rows > 0) {
        if (!x || !codes || !scales || (fmt == FP4_NVFP4 && !global_scale)) {
            set_error("null x, codes, scales or (NVFP4) global_scale");
            return FP4_ERR_INVALID_ARG;
        }
        if (((uintptr_t)x & 15) || ((uintptr_t)codes & 15) || ((uintptr_t)scales & 15) ||
            ((uintptr_t)global_scale & 3)) {
            set_error("x, codes and scales must be 16-byte aligned, global_scale 4-byte aligned");
            return FP4_ERR_ALIGNMENT;
        }
    }
    fp4_status st = check_arch();
    if (st != FP4_OK) return st;
    if (rows == 0) return FP4_OK;

    float* scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != FP4_OK) return st;

    cudaStream_t s = (cudaStream_t)stream;
    QuantLaunch q;
    q.fmt = fmt;
    q.x = static_cast<const uint16_t*>(x);
    q.x_ld = k;
    q.rows = rows;
    q.rows_pad = round_up(rows, 128);
    q.k = k;
    q.codes = static_cast<uint8_t*>(codes);
    q.scales = static_cast<uint8_t*>(scales);
    q.global_out = global_scale;
    if (fmt == FP4_NVFP4 && mode == FP4_SCALE_DYNAMIC) {
        const int np = amax_partials_count(rows * k);
        if (np > kNoAllocSlots) {
            set_error("the amax pass needs %d partial slots but the static scratch holds %d", np, kNoAllocSlots);
            return FP4_ERR_WORKSPACE;
        }
        // Every slot the quantise pass reads is written by the amax pass of the
        // same call, so nothing needs clearing.
        cudaError_t e = launch_amax_partials(q.x, rows * k, scratch, np, false, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            set_error("amax launch: %s", cudaGetErrorString(e));
            return FP4_ERR_CUDA;
        }
        q.sg_mode = SG_PARTIALS;
        q.partials = scratch;
        q.n_partials = np;
    } else {
        q.sg_mode = SG_STATIC;
        q.static_scale = static_scale;
    }
    cudaError_t e = launch_quant(q, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_error("quantise launch: %s", cudaGetErrorString(e));
        return FP4_ERR_CUDA;
    }
    return FP4_OK;
}
