// api.cu -- the extern "C" entry points of libfp4.so (declared in fp4.h):
// argument validation, the architecture check, workspace carving and the
// launch sequence of each operation.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "mxfp8.h"
#include "w4a16.h"

namespace fp4 {

// Device-side error flags (bounded waits that gave up).  The host reaches it
// through cudaGetSymbolAddress once per device.
__device__ uint32_t g_err_word;

static thread_local char t_msg[512];

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof(t_msg), fmt, ap);
    va_end(ap);
}

static std::mutex g_dev_mtx;
static DeviceInfo g_dev[64];
static int g_arch_override = 0;
static int g_tile_policy = 0;  // fp4_set_gemm_tile_policy
static uint64_t g_wait_limit_ns = 4000000000ull;

uint64_t wait_limit_ns() { return g_wait_limit_ns; }

cudaError_t set_smem_attr_once(const void* fn, int bytes, uint64_t& done) {
    const DeviceInfo* d = current_device();
    if (!d) return cudaErrorNoDevice;
    const uint64_t bit = d->device < 64 ? (1ull << d->device) : 0ull;
    if (bit && (done & bit)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done |= bit;
    return e;
}

const DeviceInfo* current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_dev_mtx);
    DeviceInfo& d = g_dev[dev];
    if (d.device < 0) {
        int major = 0, minor = 0, sms = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        void* p = nullptr;
        if (major * 10 + minor == 103) {
            if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) {
                cudaGetLastError();
                return nullptr;
            }
        }
        d.cc = major * 10 + minor;
        d.sm_count = sms;
        d.l2_bytes = l2;
        d.err_word = static_cast<uint32_t*>(p);
        d.device = dev;
    }
    return &d;
}

}  // namespace fp4

using namespace fp4;

// ------------------------------------------------------------ helpers

#define CHECK_OR_RETURN(cond, status, ...) \
    do {                                   \
        if (!(cond)) {                     \
            set_error(__VA_ARGS__);        \
            return (status);               \
        }                                  \
    } while (0)

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

fp4_status fp4::check_arch() {
    if (g_arch_override && g_arch_override != 103) {
        set_error("no compiled FP4 kernel for SM %d: libfp4 is built for sm_103a (GB300) only", g_arch_override);
        return FP4_ERR_UNSUPPORTED_ARCH;
    }
    const DeviceInfo* d = current_device();
    CHECK_OR_RETURN(d != nullptr, FP4_ERR_CUDA, "no usable CUDA device");
    CHECK_OR_RETURN(d->cc == 103, FP4_ERR_UNSUPPORTED_ARCH,
                    "no compiled FP4 kernel for SM %d: libfp4 is built for sm_103a (GB300) only", d->cc);
    return FP4_OK;
}

static fp4_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return FP4_OK;
    set_error("%s: %s", what, cudaGetErrorString(e));
    cudaGetLastError();
    return FP4_ERR_CUDA;
}

static fp4_status check_fmt(int fmt) {
    CHECK_OR_RETURN(fmt == FP4_NVFP4 || fmt == FP4_MXFP4, FP4_ERR_INVALID_ARG, "unknown format %d", fmt);
    return FP4_OK;
}

static fp4_status check_k(int64_t k) {
    CHECK_OR_RETURN(k > 0 && k % 32 == 0 && k < (1ll << 31), FP4_ERR_SHAPE,
                    "k = %lld must be a positive multiple of 32", (long long)k);
    return FP4_OK;
}

static fp4_status check_rows(int64_t r, const char* name) {
    CHECK_OR_RETURN(r >= 0 && r < (1ll << 31), FP4_ERR_SHAPE, "%s = %lld out of range", name, (long long)r);
    return FP4_OK;
}

static fp4_status check_static(int fmt, int mode, float s) {
    CHECK_OR_RETURN(mode == FP4_SCALE_DYNAMIC || mode == FP4_SCALE_STATIC, FP4_ERR_INVALID_ARG,
                    "unknown scale mode %d", mode);
    if (mode == FP4_SCALE_STATIC) {
        CHECK_OR_RETURN(fmt == FP4_NVFP4, FP4_ERR_INVALID_ARG, "MXFP4 has no global scale: use FP4_SCALE_DYNAMIC");
        CHECK_OR_RETURN(isfinite(s) && s > 0.0f, FP4_ERR_INVALID_SCALE,
                        "static activation scale %g is not finite and > 0 (a missing checkpoint scale must not "
                        "become zero)",
                        (double)s);
    }
    return FP4_OK;
}

#define TRY(x)                           \
    do {                                 \
        fp4_status _s = (x);             \
        if (_s != FP4_OK) return _s;     \
    } while (0)

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ------------------------------------------------------------ utilities

extern "C" int fp4_abi_version(void) { return FP4_ABI_VERSION; }

extern "C" const char* fp4_status_string(int s) {
    switch (s) {
        case FP4_OK: return "FP4_OK";
        case FP4_ERR_INVALID_ARG: return "FP4_ERR_INVALID_ARG";
        case FP4_ERR_SHAPE: return "FP4_ERR_SHAPE";
        case FP4_ERR_ALIGNMENT: return "FP4_ERR_ALIGNMENT";
        case FP4_ERR_UNSUPPORTED_ARCH: return "FP4_ERR_UNSUPPORTED_ARCH";
        case FP4_ERR_MISSING_SCALE: return "FP4_ERR_MISSING_SCALE";
        case FP4_ERR_INVALID_SCALE: return "FP4_ERR_INVALID_SCALE";
        case FP4_ERR_WORKSPACE: return "FP4_ERR_WORKSPACE";
        case FP4_ERR_CUDA: return "FP4_ERR_CUDA";
        case FP4_ERR_DEVICE_TIMEOUT: return "FP4_ERR_DEVICE_TIMEOUT";
    }
    return "FP4_ERR_UNKNOWN";
}

extern "C" const char* fp4_last_error_message(void) { return t_msg; }

extern "C" size_t fp4_codes_bytes(int64_t rows, int64_t k) {
    if (rows < 0 || k < 0) return 0;
    return (size_t)rows * (size_t)(k / 2);
}

extern "C" size_t fp4_scales_bytes(int fmt, int64_t rows, int64_t k) {
    if (rows < 0 || k < 0 || (fmt != FP4_NVFP4 && fmt != FP4_MXFP4)) return 0;
    const int blk = fmt == FP4_NVFP4 ? 16 : 32;
    return (size_t)round_up(rows, 128) * (size_t)sf_cols_padded(k, blk);
}

extern "C" void fp4_set_arch_override(int sm) { g_arch_override = sm; }

extern "C" fp4_status fp4_set_gemm_tile_policy(int policy) {
    CHECK_OR_RETURN(policy >= 0 && policy <= 5, FP4_ERR_INVALID_ARG, "tile policy %d not in 0..5", policy);
    g_tile_policy = policy;
    return FP4_OK;
}

extern "C" fp4_status fp4_device_status(void* stream) {
    TRY(check_arch());
    const DeviceInfo* d = current_device();
    TRY(cuda_status(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize"));
    uint32_t v = 0;
    TRY(cuda_status(cudaMemcpy(&v, d->err_word, 4, cudaMemcpyDeviceToHost), "reading device flags"));
    if (v) {
        const uint32_t zero = 0;
        TRY(cuda_status(cudaMemcpy(d->err_word, &zero, 4, cudaMemcpyHostToDevice), "clearing device flags"));
        set_error("a device-side wait gave up (flags 0x%x)", v);
        return FP4_ERR_DEVICE_TIMEOUT;
    }
    return FP4_OK;
}

// A barrier that nothing completes: the wait must give up by itself.
__global__ void timeout_probe_kernel(WaitCfg wc) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, wc, &abort_flag);
    __syncthreads();
}

extern "C" fp4_status fp4_debug_timeout_probe(int64_t limit_us, void* stream) {
    CHECK_OR_RETURN(limit_us > 0 && limit_us <= 1000000, FP4_ERR_INVALID_ARG, "limit_us must be in (0, 1e6]");
    TRY(check_arch());
    const DeviceInfo* d = current_device();
    WaitCfg wc;
    wc.limit_ns = (uint64_t)limit_us * 1000ull;
    wc.err = d->err_word;
    timeout_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(wc);
    return cuda_status(cudaGetLastError(), "timeout probe launch");
}

// --------------------------------------------------------- quantiser

extern "C" size_t fp4_quantize_workspace_size(int fmt, int64_t rows, int64_t k) {
    (void)rows;
    (void)k;
    return fmt == FP4_NVFP4 ? 4096 : 0;
}

// Enqueue the quantisation of x [rows, k]; ws holds the amax partials.
static fp4_status enqueue_quantize(int fmt, const void* x, int64_t rows, int64_t k, int mode, float st, void* codes,
                                   void* scales, float* gscale, float* partials, bool pdl, cudaStream_t s) {
    QuantLaunch q;
    q.fmt = fmt;
    q.x = static_cast<const uint16_t*>(x);
    q.x_ld = k;
    q.rows = rows;
    q.rows_pad = round_up(rows, 128);
    q.k = k;
    q.codes = static_cast<uint8_t*>(codes);
    q.scales = static_cast<uint8_t*>(scales);
    q.global_out = gscale;
    q.pdl = pdl;
    if (fmt == FP4_NVFP4 && mode == FP4_SCALE_DYNAMIC) {
        const int np = amax_partials_count(rows * k);
        TRY(cuda_status(launch_amax_partials(q.x, rows * k, partials, np, pdl, s), "amax launch"));
        q.sg_mode = SG_PARTIALS;
        q.partials = partials;
        q.n_partials = np;
        // the quantiser depends on the abs-max pass alone, which starts only after
        // x is complete: it may start early and load its first rows before its wait
        q.pdl = true;
        q.x_before_wait = true;
    } else {
        q.sg_mode = SG_STATIC;
        q.static_scale = st;
    }
    return cuda_status(launch_quant(q, s), "quantise launch");
}

static fp4_status validate_quantize(int fmt, const void* x, int64_t rows, int64_t k, int mode, float st,
                                    void* codes, void* scales, float* gscale, void* ws, size_t wsb) {
    TRY(check_fmt(fmt));
    TRY(check_rows(rows, "rows"));
    TRY(check_k(k));
    TRY(check_static(fmt, mode, st));
    if (rows == 0) return FP4_OK;  // nothing is read or written
    CHECK_OR_RETURN(x && codes && scales, FP4_ERR_INVALID_ARG, "null x, codes or scales");
    CHECK_OR_RETURN(fmt == FP4_MXFP4 || gscale, FP4_ERR_INVALID_ARG, "NVFP4 needs a global_scale output");
    CHECK_OR_RETURN(aligned16(x) && aligned16(codes) && aligned16(scales) && aligned4(gscale), FP4_ERR_ALIGNMENT,
                    "x, codes and scales must be 16-byte aligned, global_scale 4-byte aligned");
    const size_t need = fp4_quantize_workspace_size(fmt, rows, k);
    CHECK_OR_RETURN(wsb >= need && (need == 0 || (ws && aligned16(ws))), FP4_ERR_WORKSPACE,
                    "workspace %zu bytes, need %zu (16-byte aligned)", wsb, need);
    return FP4_OK;
}

extern "C" fp4_status fp4_quantize_act(int fmt, const void* x, int64_t rows, int64_t k, int mode, float st,
                                       void* codes, void* scales, float* gscale, void* ws, size_t wsb,
                                       void* stream) {
    TRY(validate_quantize(fmt, x, rows, k, mode, st, codes, scales, gscale, ws, wsb));
    TRY(check_arch());
    if (rows == 0) return FP4_OK;
    return enqueue_quantize(fmt, x, rows, k, mode, st, codes, scales, gscale, static_cast<float*>(ws), false,
                            (cudaStream_t)stream);
}

extern "C" fp4_status fp4_prepack_weight(int fmt, const void* w, int64_t n, int64_t k, void* codes, void* scales,
                                         float* gscale, void* ws, size_t wsb, void* stream) {
    return fp4_quantize_act(fmt, w, n, k, FP4_SCALE_DYNAMIC, 0.0f, codes, scales, gscale, ws, wsb, stream);
}

// ------------------------------------------------------------- GEMM

static const int64_t kDecodeMaxM = 64;

struct GemmPlan {
    bool decode;
    bool pair;  // CTA-pair kernel (256 x 256 tiles)
    bool mc;    // one-CTA kernel in clusters of two sharing each 256-row weight tile (TMA multicast)
    int bn;
    int splits;
};

static GemmPlan plan_gemm(int64_t m, int64_t n, int64_t k, int sms) {
    GemmPlan p;
    p.pair = false;
    p.mc = false;
    const int64_t kbt = gemm_k_blocks(k);
    if (m <= kDecodeMaxM) {
        // decode, swap-AB: the weights are the MMA's M side (128-row tiles), the
        // m activation rows its N side (32 or 64, rows past m zero-filled by
        // the TMA), split-K so that about three units land on every SM;
        // deterministic reduction afterwards
        p.decode = true;
        p.bn = m <= 32 ? 32 : 64;
        const int64_t qtiles = (n + 127) / 128;
        // with weight tiles for at least half the SMs, one K range per tile
        // (no partials, no reduction launch); fewer tiles are split along K
        int64_t s = 2 * qtiles >= sms ? 1 : (3 * (int64_t)sms + qtiles - 1) / qtiles;
        if (s > kbt / 2) s = kbt / 2;
        if (s > 16) s = 16;
        if (s < 1) s = 1;
        // make every split non-empty
        const int64_t per = (kbt + s - 1) / s;
        s = (kbt + per - 1) / per;
        p.splits = (int)s;
    } else {
        p.decode = false;
        // persistent CTAs take whole tiles, so a launch lasts about (waves of
        // tiles) x (tile time); a 256-wide tile takes about 1.5x a 128-wide one
        // (96 KB against 64 KB of shared-memory traffic per K block, which
        // bounds both)
        const int64_t w256 = (((m + 127) / 128) * ((n + 255) / 256) + sms - 1) / sms;
        const int64_t w128 = (((m + 127) / 128) * ((n + 127) / 128) + sms - 1) / sms;
        p.bn = 3 * w256 <= 2 * w128 ? 256 : 128;
        p.splits = 1;
        // The CTA-pair kernel is opt-in: on the 8192 x 14336 x 4096 prefill it
        // runs within a few percent of the one-CTA kernel (151-157 against
        // 156-159 us), since each SM's tensor core still takes in the peer's
        // half of the 256-wide operand tile, so an SM's operand stream per K
        // block barely shrinks.
        p.pair = g_tile_policy == 2 && m >= 256 && n >= 256;
        // weight-tile sharing pairs: 256-wide tiles, whole pairs of 128-row
        // activation tiles, and enough pair units for every cluster
        const int64_t mt = (m + 127) / 128;
        p.mc = g_tile_policy == 5 && p.bn == 256 && mt % 2 == 0 && (mt / 2) * ((n + 255) / 256) >= sms / 2;
    }
    return p;
}

// fp4_gemm's choice of the fused decode kernel (activation quantisation
// inside the GEMM launch): automatic for m <= kDecodeFusedAutoMaxM when the
// weight has tiles for at least half the SMs, forced by tile policy 3.
static bool use_fused_decode(int64_t m, int64_t n, int64_t k, int sms) {
    const bool want = g_tile_policy == 3 ||
                      (g_tile_policy == 0 && m <= kDecodeFusedAutoMaxM && (n + 127) / 128 >= (int64_t)sms / 2);
    return m <= kDecodeFusedMaxM && k <= kDecodeFusedMaxK && want;
}

extern "C" fp4_status fp4_debug_plan_gemm(int64_t m, int64_t n, int64_t k, int sm_count, int64_t* out,
                                          int max_out) {
    CHECK_OR_RETURN(m > 0 && n > 0 && k > 0 && sm_count > 0 && out && max_out >= 5, FP4_ERR_INVALID_ARG,
                    "plan query needs positive sizes, an SM count and room for 5 entries");
    const GemmPlan p = plan_gemm(m, n, k, sm_count);
    out[0] = p.decode ? 1 : 0;
    out[1] = p.bn;
    out[2] = p.splits;
    out[3] = p.pair ? 1 : 0;
    out[4] = use_fused_decode(m, n, k, sm_count) ? 1 : 0;
    if (max_out >= 6) out[5] = p.mc ? 1 : 0;
    return FP4_OK;
}

static size_t gemm_prequant_ws(int64_t m, int64_t n, int64_t k, int sms) {
    GemmPlan p = plan_gemm(m, n, k, sms);
    if (p.decode && p.splits > 1) return align256((size_t)p.splits * (size_t)m * (size_t)n * 4);
    return 0;
}

static int sms_for_sizing() {
    const DeviceInfo* d = current_device();
    return d ? d->sm_count : 160;  // sizing without a device: an upper bound on the SM count
}

extern "C" size_t fp4_gemm_prequant_workspace_size(int fmt, int64_t m, int64_t n, int64_t k) {
    (void)fmt;
    if (m <= 0 || n <= 0 || k <= 0) return 0;
    // Take the larger of the plans for this device and for a 160-SM upper bound.
    size_t a = gemm_prequant_ws(m, n, k, sms_for_sizing());
    size_t b = gemm_prequant_ws(m, n, k, 160);
    return a > b ? a : b;
}

extern "C" size_t fp4_gemm_workspace_size(int fmt, int64_t m, int64_t n, int64_t k) {
    if (m < 0 || n < 0 || k <= 0) return 0;
    size_t s = align256(fp4_codes_bytes(m, k)) + align256(fp4_scales_bytes(fmt, m, k)) + 256 + 4096;
    return s + fp4_gemm_prequant_workspace_size(fmt, m, n, k);
}

static fp4_status validate_gemm_common(int fmt, int64_t m, const void* w_codes, const void* w_scales,
                                       const float* w_global, int64_t n, int64_t k, void* out) {
    TRY(check_fmt(fmt));
    TRY(check_rows(m, "m"));
    TRY(check_rows(n, "n"));
    TRY(check_k(k));
    CHECK_OR_RETURN(n % 8 == 0, FP4_ERR_SHAPE, "n = %lld must be a multiple of 8", (long long)n);
    if (m == 0 || n == 0) return FP4_OK;  // nothing is read or written
    CHECK_OR_RETURN(w_codes && w_scales && out, FP4_ERR_INVALID_ARG, "null weight or output pointer");
    CHECK_OR_RETURN(fmt == FP4_MXFP4 || w_global, FP4_ERR_MISSING_SCALE, "NVFP4 weight global scale is NULL");
    CHECK_OR_RETURN(aligned16(w_codes) && aligned16(w_scales) && aligned16(out) && aligned4(w_global),
                    FP4_ERR_ALIGNMENT, "weights / output must be 16-byte aligned, global scales 4-byte aligned");
    return FP4_OK;
}

// GEMM on quantised operands A [m, k] and W [n, k]; part = split-K workspace.
static fp4_status enqueue_gemm(int fmt, const uint8_t* ac, const uint8_t* as, const float* ag, int64_t m,
                               const uint8_t* wc, const uint8_t* wsc, const float* wg, int64_t n, int64_t k,
                               void* out, float* part, bool pdl, cudaStream_t s) {
    const DeviceInfo* d = current_device();
    GemmPlan p = plan_gemm(m, n, k, d->sm_count);
    GemmLaunch g;
    g.fmt = fmt;
    g.k = k;
    g.pdl = pdl;
    g.bn = p.bn;
    if (!p.decode) {
        g.epi = EPI_BF16;
        g.p_codes = ac, g.p_scales = as, g.p_rows = m, g.p_rows_valid = m, g.p_global = ag;
        g.q_codes = wc, g.q_scales = wsc, g.q_rows = n, g.q_rows_valid = n, g.q_global = wg;
        g.out = out;
        g.ldo = n;
        g.early_q = true;  // weights
        g.mc = p.mc;
        if (p.pair) return cuda_status(launch_gemm_pair(g, s), "GEMM launch");
        return cuda_status(launch_gemm(g, s), "GEMM launch");
    }
    // decode: weights on the MMA M side, activations on N, split-K partials
    // part[split][m][n] (the transposed epilogues write token-major rows)
    g.p_codes = wc, g.p_scales = wsc, g.p_rows = n, g.p_rows_valid = n, g.p_global = wg;
    g.q_codes = ac, g.q_scales = as, g.q_rows = m, g.q_rows_valid = m, g.q_global = ag;
    g.splits = p.splits;
    g.early_p = true;  // weights
    if (p.splits == 1) {
        g.epi = EPI_BF16_T;
        g.out = out;
        g.ldo = n;
        return cuda_status(launch_gemm(g, s), "GEMM launch");
    }
    g.epi = EPI_PARTIAL_T;
    g.out = part;
    g.ldo = n;
    TRY(cuda_status(launch_gemm(g, s), "GEMM launch"));
    return cuda_status(launch_splitk_reduce(part, p.splits, m, n, ag, wg, fmt == FP4_MXFP4,
                                            static_cast<uint16_t*>(out), pdl, s),
                       "split-K reduce launch");
}

extern "C" fp4_status fp4_gemm_prequant(int fmt, const void* a_codes, const void* a_scales, const float* a_global,
                                        int64_t m, const void* w_codes, const void* w_scales, const float* w_global,
                                        int64_t n, int64_t k, void* out, void* ws, size_t wsb, void* stream) {
    TRY(validate_gemm_common(fmt, m, w_codes, w_scales, w_global, n, k, out));
    if (m == 0 || n == 0) return check_arch();
    CHECK_OR_RETURN(a_codes && a_scales, FP4_ERR_INVALID_ARG, "null activation codes or scales");
    CHECK_OR_RETURN(fmt == FP4_MXFP4 || a_global, FP4_ERR_MISSING_SCALE, "NVFP4 activation global scale is NULL");
    CHECK_OR_RETURN(aligned16(a_codes) && aligned16(a_scales) && aligned4(a_global), FP4_ERR_ALIGNMENT,
                    "activation codes / scales must be 16-byte aligned");
    const size_t need = fp4_gemm_prequant_workspace_size(fmt, m, n, k);
    CHECK_OR_RETURN(wsb >= need && (need == 0 || (ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0)),
                    FP4_ERR_WORKSPACE, "workspace %zu bytes, need %zu (256-byte aligned)", wsb, need);
    TRY(check_arch());
    if (m == 0 || n == 0) return FP4_OK;
    return enqueue_gemm(fmt, static_cast<const uint8_t*>(a_codes), static_cast<const uint8_t*>(a_scales), a_global,
                        m, static_cast<const uint8_t*>(w_codes), static_cast<const uint8_t*>(w_scales), w_global, n,
                        k, out, static_cast<float*>(ws), false, (cudaStream_t)stream);
}

static fp4_status check_mx_elem(int elem) {
    CHECK_OR_RETURN(elem >= FP4_MX_E4M3 && elem <= FP4_MX_E3M2, FP4_ERR_INVALID_ARG, "unknown MX element format %d",
                    elem);
    return FP4_OK;
}

extern "C" fp4_status fp4_quantize_mx(int elem, const void* x, int64_t rows, int64_t k, void* codes, void* scales,
                                      void* stream) {
    TRY(check_mx_elem(elem));
    TRY(check_rows(rows, "rows"));
    TRY(check_k(k));
    if (rows == 0) return check_arch();
    CHECK_OR_RETURN(x && codes && scales, FP4_ERR_INVALID_ARG, "null input, codes or scales pointer");
    CHECK_OR_RETURN(aligned16(x) && aligned16(codes) && aligned16(scales), FP4_ERR_ALIGNMENT,
                    "input, codes and scales must be 16-byte aligned");
    TRY(check_arch());
    const DeviceInfo* d = current_device();
    return cuda_status(launch_mx8_quant(elem, static_cast<const uint16_t*>(x), rows, k, static_cast<uint8_t*>(codes),
                                        static_cast<uint8_t*>(scales), d->sm_count, (cudaStream_t)stream),
                       "MX quantise launch");
}

extern "C" fp4_status fp4_quantize_mxfp8(const void* x, int64_t rows, int64_t k, void* codes, void* scales,
                                         void* stream) {
    return fp4_quantize_mx(FP4_MX_E4M3, x, rows, k, codes, scales, stream);
}

// Type code of an MXFP8 element format in the kind::mxf8f6f4 instruction descriptor.
static int mx8_type_code(int elem) { return elem == FP4_MX_E4M3 ? 0 : 1; }

static fp4_status validate_gemm_mx(int a_elem, int64_t m, int w_elem, const void* w_codes, const void* w_scales,
                                   int64_t n, int64_t k, void* out, bool fp6_a_ok) {
    TRY(check_mx_elem(a_elem));
    TRY(check_mx_elem(w_elem));
    CHECK_OR_RETURN((a_elem <= FP4_MX_E5M2 || fp6_a_ok) && w_elem <= FP4_MX_E5M2, FP4_ERR_INVALID_ARG,
                    "the MX GEMM reads E4M3 / E5M2 codes: widen MXFP6 codes first (fp4_mx_widen)");
    TRY(check_rows(m, "m"));
    TRY(check_rows(n, "n"));
    TRY(check_k(k));
    CHECK_OR_RETURN(n % 8 == 0, FP4_ERR_SHAPE, "n = %lld must be a multiple of 8", (long long)n);
    if (m == 0 || n == 0) return FP4_OK;
    CHECK_OR_RETURN(w_codes && w_scales && out, FP4_ERR_INVALID_ARG, "null weight or output pointer");
    CHECK_OR_RETURN(aligned16(w_codes) && aligned16(w_scales) && aligned16(out), FP4_ERR_ALIGNMENT,
                    "weights / output must be 16-byte aligned");
    return FP4_OK;
}

// MX GEMM with 8-bit-container operands: the one-CTA kernel with the bf16
// epilogue for every m (tile width by the same wave rule as FP4).
static fp4_status enqueue_gemm_mx(int a_elem, const uint8_t* ac, const uint8_t* as, int64_t m, int w_elem,
                                  const uint8_t* wc, const uint8_t* wsc, int64_t n, int64_t k, void* out, bool pdl,
                                  cudaStream_t s) {
    const DeviceInfo* d = current_device();
    const int64_t sms = d->sm_count;
    const int64_t w256 = (((m + 127) / 128) * ((n + 255) / 256) + sms - 1) / sms;
    const int64_t w128 = (((m + 127) / 128) * ((n + 127) / 128) + sms - 1) / sms;
    GemmLaunch g;
    g.fmt = FMT_MX8;
    g.p_type = mx8_type_code(a_elem);
    g.q_type = mx8_type_code(w_elem);
    g.k = k;
    g.pdl = pdl;
    g.bn = 3 * w256 <= 2 * w128 ? 256 : 128;
    g.epi = EPI_BF16;
    g.p_codes = ac, g.p_scales = as, g.p_rows = m, g.p_rows_valid = m;
    g.q_codes = wc, g.q_scales = wsc, g.q_rows = n, g.q_rows_valid = n;
    g.out = out;
    g.ldo = n;
    g.early_q = true;  // weights
    return cuda_status(launch_gemm(g, s), "MX GEMM launch");
}

extern "C" fp4_status fp4_gemm_mx_prequant(int a_elem, const void* a_codes, const void* a_scales, int64_t m,
                                           int w_elem, const void* w_codes, const void* w_scales, int64_t n,
                                           int64_t k, void* out, void* stream) {
    TRY(validate_gemm_mx(a_elem, m, w_elem, w_codes, w_scales, n, k, out, false));
    if (m == 0 || n == 0) return check_arch();
    CHECK_OR_RETURN(a_codes && a_scales, FP4_ERR_INVALID_ARG, "null activation codes or scales");
    CHECK_OR_RETURN(aligned16(a_codes) && aligned16(a_scales), FP4_ERR_ALIGNMENT,
                    "activation codes / scales must be 16-byte aligned");
    TRY(check_arch());
    return enqueue_gemm_mx(a_elem, static_cast<const uint8_t*>(a_codes), static_cast<const uint8_t*>(a_scales), m,
                           w_elem, static_cast<const uint8_t*>(w_codes), static_cast<const uint8_t*>(w_scales), n, k,
                           out, false, (cudaStream_t)stream);
}

extern "C" fp4_status fp4_mx_widen(int elem, const void* codes, int64_t rows, int64_t k, void* out, void* stream) {
    TRY(check_mx_elem(elem));
    CHECK_OR_RETURN(elem >= FP4_MX_E2M3, FP4_ERR_INVALID_ARG, "only MXFP6 codes (E2M3 / E3M2) are widened");
    TRY(check_rows(rows, "rows"));
    TRY(check_k(k));
    if (rows == 0) return check_arch();
    CHECK_OR_RETURN(codes && out, FP4_ERR_INVALID_ARG, "null codes or output pointer");
    CHECK_OR_RETURN(aligned16(codes) && aligned16(out), FP4_ERR_ALIGNMENT, "codes and output must be 16-byte aligned");
    TRY(check_arch());
    const DeviceInfo* d = current_device();
    return cuda_status(launch_mx6_widen(elem, static_cast<const uint8_t*>(codes), static_cast<uint8_t*>(out), rows * k,
                                        d->sm_count, (cudaStream_t)stream),
                       "MX widen launch");
}

extern "C" size_t fp4_gemm_mx_workspace_size(int64_t m, int64_t k) {
    if (m < 0 || k <= 0) return 0;
    return align256((size_t)m * (size_t)k) + align256(fp4_scales_bytes(FP4_MXFP4, m, k));
}

extern "C" fp4_status fp4_gemm_mx(int a_elem, const void* x, int64_t m, int w_elem, const void* w_codes,
                                  const void* w_scales, int64_t n, int64_t k, void* out, void* ws, size_t wsb,
                                  void* stream) {
    TRY(validate_gemm_mx(a_elem, m, w_elem, w_codes, w_scales, n, k, out, true));
    if (m == 0 || n == 0) return check_arch();
    CHECK_OR_RETURN(x, FP4_ERR_INVALID_ARG, "null activation pointer");
    CHECK_OR_RETURN(aligned16(x), FP4_ERR_ALIGNMENT, "activations must be 16-byte aligned");
    const size_t need = fp4_gemm_mx_workspace_size(m, k);
    CHECK_OR_RETURN(wsb >= need && ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0, FP4_ERR_WORKSPACE,
                    "workspace %zu bytes, need %zu (256-byte aligned)", wsb, need);
    TRY(check_arch());
    uint8_t* ac = static_cast<uint8_t*>(ws);
    uint8_t* as = ac + align256((size_t)m * (size_t)k);
    const DeviceInfo* d = current_device();
    cudaStream_t s = (cudaStream_t)stream;
    // MXFP6 activations: quantised to the 6-bit format, stored as the E4M3
    // codes of the same values (exact), and multiplied as E4M3
    const bool fp6 = a_elem >= FP4_MX_E2M3;
    TRY(cuda_status(launch_mx8_quant(a_elem, static_cast<const uint16_t*>(x), m, k, ac, as, d->sm_count, s, fp6),
                    "MX quantise launch"));
    return enqueue_gemm_mx(fp6 ? FP4_MX_E4M3 : a_elem, ac, as, m, w_elem, static_cast<const uint8_t*>(w_codes),
                           static_cast<const uint8_t*>(w_scales), n, k, out, true, s);
}

extern "C" fp4_status fp4_gemm_w4a16(int fmt, const void* x, int64_t m, const void* w_codes, const void* w_scales,
                                     const float* w_global, int64_t n, int64_t k, void* out, void* stream) {
    TRY(validate_gemm_common(fmt, m, w_codes, w_scales, w_global, n, k, out));
    CHECK_OR_RETURN(m <= kW4A16MaxM, FP4_ERR_SHAPE, "m = %lld: the weight-only path takes at most %d rows",
                    (long long)m, kW4A16MaxM);
    CHECK_OR_RETURN(k <= kW4A16MaxK, FP4_ERR_SHAPE, "k = %lld: the weight-only path takes k <= %d", (long long)k,
                    kW4A16MaxK);
    if (m == 0 || n == 0) return check_arch();
    CHECK_OR_RETURN(x, FP4_ERR_INVALID_ARG, "null activation pointer");
    CHECK_OR_RETURN(aligned16(x), FP4_ERR_ALIGNMENT, "activations must be 16-byte aligned");
    TRY(check_arch());
    const DeviceInfo* d = current_device();
    const int sms = d ? d->sm_count : 148;
    // the tensor-core kernel takes one CTA per 128 weight rows and runs at a
    // near-constant time paced by its 256 small (N = 16) MMAs per CTA: automatic
    // for 3-4 activation rows when the tiles fill at least half the SMs (the
    // CUDA-core kernel's time grows with the rows, the tensor-core one's does not)
    const bool tc = g_tile_policy == 4 || (g_tile_policy == 0 && m >= 3 && 2 * ((n + 127) / 128) >= sms);
    auto launch = tc ? launch_w4a16_tc : launch_w4a16;
    return cuda_status(launch(fmt, static_cast<const uint16_t*>(x), (int)m, n, k, static_cast<const uint8_t*>(w_codes),
                              static_cast<const uint8_t*>(w_scales), w_global, static_cast<uint16_t*>(out),
                              (cudaStream_t)stream),
                       "weight-only launch");
}

extern "C" fp4_status fp4_gemm(int fmt, const void* x, int64_t m, int mode, float st, const void* w_codes,
                               const void* w_scales, const float* w_global, int64_t n, int64_t k, void* out,
                               void* ws, size_t wsb, void* stream) {
    TRY(validate_gemm_common(fmt, m, w_codes, w_scales, w_global, n, k, out));
    TRY(check_static(fmt, mode, st));
    if (m == 0 || n == 0) return check_arch();
    CHECK_OR_RETURN(x, FP4_ERR_INVALID_ARG, "null activation pointer");
    CHECK_OR_RETURN(aligned16(x), FP4_ERR_ALIGNMENT, "activations must be 16-byte aligned");
    const size_t need = fp4_gemm_workspace_size(fmt, m, n, k);
    CHECK_OR_RETURN(wsb >= need && ws && (reinterpret_cast<uintptr_t>(ws) & 255) == 0, FP4_ERR_WORKSPACE,
                    "workspace %zu bytes, need %zu (256-byte aligned)", wsb, need);
    TRY(check_arch());
    if (m == 0 || n == 0) return FP4_OK;
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t* ac = base;
    base += align256(fp4_codes_bytes(m, k));
    uint8_t* as = base;
    base += align256(fp4_scales_bytes(fmt, m, k));
    float* ag = reinterpret_cast<float*>(base);
    const DeviceInfo* d = current_device();
    if (use_fused_decode(m, n, k, d->sm_count)) {
        // decode: one launch (in-kernel activation quantisation, one CTA per
        // 128 weight rows, no split-K); the activation s_g goes to the workspace
        return cuda_status(launch_decode_fused(fmt, static_cast<const uint16_t*>(x), (int)m, n, k,
                                               static_cast<const uint8_t*>(w_codes),
                                               static_cast<const uint8_t*>(w_scales), w_global,
                                               mode == FP4_SCALE_DYNAMIC ? 1 : 0, st, ag,
                                               static_cast<uint16_t*>(out), false, (cudaStream_t)stream),
                           "decode launch");
    }
    base += 256;
    float* partials = reinterpret_cast<float*>(base);
    base += 4096;
    float* part = reinterpret_cast<float*>(base);
    cudaStream_t s = (cudaStream_t)stream;
    TRY(enqueue_quantize(fmt, x, m, k, mode, st, ac, as, ag, partials, false, s));
    return enqueue_gemm(fmt, ac, as, ag, m, static_cast<const uint8_t*>(w_codes),
                        static_cast<const uint8_t*>(w_scales), w_global, n, k, out, part, true, s);
}
