"""Python binding of libfp4.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module only
allocates outputs / workspaces with PyTorch, passes raw device pointers and
the current CUDA stream, and turns status codes into exceptions.  If the
in-tree library is missing it raises: there is no fallback implementation.

The raw C entry points are re-exported under their C names (``fp4_gemm``,
``fp4_quantize_act``, ...) taking integers (pointers, sizes); the helpers
below them take tensors.
"""
import ctypes
import os

import torch

NVFP4 = 0
MXFP4 = 1
DYNAMIC = 0
STATIC = 1
BLOCK = {NVFP4: 16, MXFP4: 32}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp4.so")

STATUS = {
    0: "FP4_OK", 1: "FP4_ERR_INVALID_ARG", 2: "FP4_ERR_SHAPE", 3: "FP4_ERR_ALIGNMENT",
    4: "FP4_ERR_UNSUPPORTED_ARCH", 5: "FP4_ERR_MISSING_SCALE", 6: "FP4_ERR_INVALID_SCALE",
    7: "FP4_ERR_WORKSPACE", 8: "FP4_ERR_CUDA", 9: "FP4_ERR_DEVICE_TIMEOUT",
}
STATUS_CODE = {v: k for k, v in STATUS.items()}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_INT = ctypes.c_int

# name -> (restype, argtypes)
_SIGNATURES = {
    "fp4_abi_version": (_INT, []),
    "fp4_status_string": (ctypes.c_char_p, [_INT]),
    "fp4_last_error_message": (ctypes.c_char_p, []),
    "fp4_codes_bytes": (_SZ, [_I64, _I64]),
    "fp4_scales_bytes": (_SZ, [_INT, _I64, _I64]),
    "fp4_device_status": (_INT, [_P]),
    "fp4_set_arch_override": (None, [_INT]),
    "fp4_set_gemm_tile_policy": (_INT, [_INT]),
    "fp4_set_moe_policy": (_INT, [_INT]),
    "fp4_debug_timeout_probe": (_INT, [_I64, _P]),
    "fp4_debug_plan_gemm": (_INT, [_I64, _I64, _I64, _INT, ctypes.POINTER(ctypes.c_int64), _INT]),
    "fp4_quantize_workspace_size": (_SZ, [_INT, _I64, _I64]),
    "fp4_quantize_act": (_INT, [_INT, _P, _I64, _I64, _INT, _F, _P, _P, _P, _P, _SZ, _P]),
    "fp4_quantize_act_noalloc": (_INT, [_INT, _P, _I64, _I64, _INT, _F, _P, _P, _P, _P]),
    "fp4_prepack_weight": (_INT, [_INT, _P, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "fp4_gemm_workspace_size": (_SZ, [_INT, _I64, _I64, _I64]),
    "fp4_gemm": (_INT, [_INT, _P, _I64, _INT, _F, _P, _P, _P, _I64, _I64, _P, _P, _SZ, _P]),
    "fp4_gemm_prequant_workspace_size": (_SZ, [_INT, _I64, _I64, _I64]),
    "fp4_gemm_prequant": (_INT, [_INT, _P, _P, _P, _I64, _P, _P, _P, _I64, _I64, _P, _P, _SZ, _P]),
    "fp4_gemm_w4a16": (_INT, [_INT, _P, _I64, _P, _P, _P, _I64, _I64, _P, _P]),
    "fp4_quantize_mxfp8": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "fp4_quantize_mx": (_INT, [_INT, _P, _I64, _I64, _P, _P, _P]),
    "fp4_gemm_mx_prequant": (_INT, [_INT, _P, _P, _I64, _INT, _P, _P, _I64, _I64, _P, _P]),
    "fp4_gemm_mx_workspace_size": (_SZ, [_I64, _I64]),
    "fp4_mx_widen": (_INT, [_INT, _P, _I64, _I64, _P, _P]),
    "fp4_gemm_mx": (_INT, [_INT, _P, _I64, _INT, _P, _P, _I64, _I64, _P, _P, _SZ, _P]),
    "fp4_moe_prepack_workspace_size": (_SZ, [_I64, _I64, _I64]),
    "fp4_moe_prepack_weights": (_INT, [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "fp4_moe_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64]),
    "fp4_moe_grouped": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                               _P, _SZ, _P]),
    "fp4_moe_workspace_layout": (_INT, [_I64, _I64, _I64, _I64, _I64, ctypes.POINTER(ctypes.c_int64), _INT]),
    "fp4_moe_grouped_stages": (_INT, [_P, _P, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, _SZ, ctypes.c_uint, _P]),
}

_lib = None


def lib():
    """Load the in-tree libfp4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfp4.so not found at %s: build it with __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGNATURES)


class FP4Error(RuntimeError):
    def __init__(self, status, msg):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__("%s: %s" % (self.name, msg))


def _check(status):
    if status != 0:
        raise FP4Error(status, lib().fp4_last_error_message().decode())


def __getattr__(name):
    # Raw C entry points under their C names.
    if name in _SIGNATURES:
        return getattr(lib(), name)
    raise AttributeError(name)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return _P(s.cuda_stream)


def _ptr(t):
    return _P(0) if t is None else _P(t.data_ptr())


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class QTensor:
    """A quantised [rows, k] tensor: codes [rows, k/2] u8, scales in the MMA
    layout (flat u8), global scale (1-element fp32; 1.0 for MXFP4)."""

    def __init__(self, fmt, rows, k, codes, scales, gscale):
        self.fmt, self.rows, self.k = fmt, rows, k
        self.codes, self.scales, self.gscale = codes, scales, gscale


def empty_qtensor(fmt, rows, k, device, n_global=1):
    L = lib()
    codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=device)
    scales = torch.empty(L.fp4_scales_bytes(fmt, rows, k), dtype=torch.uint8, device=device)
    g = torch.ones(n_global, dtype=torch.float32, device=device)
    return QTensor(fmt, rows, k, codes, scales, g)


def quantize(x, fmt=NVFP4, mode=DYNAMIC, static_scale=0.0, out=None, workspace=None, stream=None):
    """bf16 [rows, k] (CUDA) -> QTensor via fp4_quantize_act."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    rows, k = x.shape
    L = lib()
    q = out or empty_qtensor(fmt, rows, k, x.device)
    wsb = L.fp4_quantize_workspace_size(fmt, rows, k)
    ws = workspace if workspace is not None else _ws(wsb, x.device)
    _check(L.fp4_quantize_act(fmt, _ptr(x), rows, k, mode, float(static_scale), _ptr(q.codes), _ptr(q.scales),
                              _ptr(q.gscale), _ptr(ws), ws.numel(), _stream(stream)))
    return q


def prepack_weight(w, fmt=NVFP4, stream=None):
    """bf16 weight [n, k] -> QTensor (dynamic per-tensor scale), once at load."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.is_contiguous()
    n, k = w.shape
    L = lib()
    q = empty_qtensor(fmt, n, k, w.device)
    ws = _ws(L.fp4_quantize_workspace_size(fmt, n, k), w.device)
    _check(L.fp4_prepack_weight(fmt, _ptr(w), n, k, _ptr(q.codes), _ptr(q.scales), _ptr(q.gscale), _ptr(ws),
                                ws.numel(), _stream(stream)))
    return q


def gemm(x, wq, mode=DYNAMIC, static_scale=0.0, out=None, workspace=None, stream=None):
    """W4A4 linear: bf16 x [m, k] (quantised per call) times the prepacked
    weight [n, k] -> bf16 [m, n]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    m, k = x.shape
    n = wq.rows
    L = lib()
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    wsb = L.fp4_gemm_workspace_size(wq.fmt, m, n, k)
    ws = workspace if workspace is not None else _ws(wsb, x.device)
    _check(L.fp4_gemm(wq.fmt, _ptr(x), m, mode, float(static_scale), _ptr(wq.codes), _ptr(wq.scales),
                      _ptr(wq.gscale), n, k, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def gemm_prequant(aq, wq, out=None, workspace=None, stream=None):
    m, k, n = aq.rows, aq.k, wq.rows
    L = lib()
    dev = aq.codes.device
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    wsb = L.fp4_gemm_prequant_workspace_size(wq.fmt, m, n, k)
    ws = workspace if workspace is not None else (_ws(wsb, dev) if wsb else None)
    _check(L.fp4_gemm_prequant(wq.fmt, _ptr(aq.codes), _ptr(aq.scales), _ptr(aq.gscale), m, _ptr(wq.codes),
                               _ptr(wq.scales), _ptr(wq.gscale), n, k, _ptr(out), _ptr(ws),
                               0 if ws is None else ws.numel(), _stream(stream)))
    return out


def quantize_mxfp8(x, stream=None):
    """bf16 [rows, k] (CUDA) -> (codes [rows, k] uint8 E4M3, scales flat uint8
    E8M0 in the MMA layout)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    rows, k = x.shape
    L = lib()
    codes = torch.empty((rows, k), dtype=torch.uint8, device=x.device)
    scales = torch.empty(L.fp4_scales_bytes(MXFP4, rows, k), dtype=torch.uint8, device=x.device)
    _check(L.fp4_quantize_mxfp8(_ptr(x), rows, k, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales


MX_E4M3, MX_E5M2, MX_E2M3, MX_E3M2 = 0, 1, 2, 3
MX_ELEM_NAMES = {MX_E4M3: "e4m3", MX_E5M2: "e5m2", MX_E2M3: "e2m3", MX_E3M2: "e3m2"}


class MXTensor:
    """An MXFP8 / MXFP6 tensor [rows, k]: codes [rows, k] uint8 (one element
    per byte), E8M0 scales in the MMA layout (flat uint8), element format."""

    def __init__(self, elem, rows, k, codes, scales):
        self.elem, self.rows, self.k, self.codes, self.scales = elem, rows, k, codes, scales


def quantize_mx(x, elem=MX_E4M3, stream=None):
    """bf16 [rows, k] (CUDA) -> MXTensor via fp4_quantize_mx."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    rows, k = x.shape
    L = lib()
    codes = torch.empty((rows, k), dtype=torch.uint8, device=x.device)
    scales = torch.empty(L.fp4_scales_bytes(MXFP4, rows, k), dtype=torch.uint8, device=x.device)
    _check(L.fp4_quantize_mx(elem, _ptr(x), rows, k, _ptr(codes), _ptr(scales), _stream(stream)))
    return MXTensor(elem, rows, k, codes, scales)


def mx_widen(q, stream=None):
    """An MXFP6 MXTensor -> the same values as an E4M3 MXTensor (exact; the
    scales are shared), the form the MX GEMM reads."""
    codes = torch.empty_like(q.codes)
    _check(lib().fp4_mx_widen(q.elem, _ptr(q.codes), q.rows, q.k, _ptr(codes), _stream(stream)))
    return MXTensor(MX_E4M3, q.rows, q.k, codes, q.scales)


def gemm_mx_prequant(aq, wq, out=None, stream=None):
    """MX linear on quantised operands: MXTensor a [m, k] x MXTensor w [n, k] -> bf16 [m, n]."""
    m, k, n = aq.rows, aq.k, wq.rows
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=aq.codes.device)
    _check(lib().fp4_gemm_mx_prequant(aq.elem, _ptr(aq.codes), _ptr(aq.scales), m, wq.elem, _ptr(wq.codes),
                                      _ptr(wq.scales), n, k, _ptr(out), _stream(stream)))
    return out


def gemm_mx(x, wq, elem=MX_E4M3, out=None, workspace=None, stream=None):
    """MX linear: bf16 x [m, k] quantised to `elem` per call, times the
    quantised weight MXTensor [n, k] -> bf16 [m, n]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    m, k = x.shape
    n = wq.rows
    L = lib()
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    ws = workspace if workspace is not None else _ws(L.fp4_gemm_mx_workspace_size(m, k), x.device)
    _check(L.fp4_gemm_mx(elem, _ptr(x), m, wq.elem, _ptr(wq.codes), _ptr(wq.scales), n, k, _ptr(out), _ptr(ws),
                         ws.numel(), _stream(stream)))
    return out


def gemm_w4a16(x, wq, out=None, stream=None):
    """Weight-only linear: bf16 x [m, k] (m <= 4, not quantised) times the
    prepacked FP4 weight [n, k] -> bf16 [m, n]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    m, k = x.shape
    n = wq.rows
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=x.device)
    _check(lib().fp4_gemm_w4a16(wq.fmt, _ptr(x), m, _ptr(wq.codes), _ptr(wq.scales), _ptr(wq.gscale), n, k,
                                _ptr(out), _stream(stream)))
    return out


TILE_AUTO, TILE_ONE_CTA, TILE_CTA_PAIR, TILE_FUSED_DECODE, TILE_W4A16_TC, TILE_WEIGHT_PAIRS = 0, 1, 2, 3, 4, 5


def set_gemm_tile_policy(policy):
    """Choose the GEMM kernels (TILE_AUTO, TILE_ONE_CTA, TILE_CTA_PAIR, TILE_FUSED_DECODE, TILE_W4A16_TC,
    TILE_WEIGHT_PAIRS)."""
    _check(lib().fp4_set_gemm_tile_policy(int(policy)))


def plan_gemm(m, n, k, sm_count):
    """The GEMM plan for m x n x k on `sm_count` SMs (host-side query)."""
    out = (ctypes.c_int64 * 6)()
    _check(lib().fp4_debug_plan_gemm(m, n, k, sm_count, out, 6))
    return {"small_m": bool(out[0]), "bn": out[1], "splits": out[2], "pair": bool(out[3]), "fused_decode": bool(out[4]),
            "weight_pairs": bool(out[5])}


def device_status(stream=None):
    """Synchronise and raise FP4Error if a device-side wait gave up."""
    _check(lib().fp4_device_status(_stream(stream)))


# ------------------------------------------------------------------- MoE

class MoEWeights:
    def __init__(self, E, H, I, w13, w2):
        self.E, self.H, self.I = E, H, I
        self.w13, self.w2 = w13, w2  # QTensor with per-expert gscale [E]


def moe_prepack(w13, w2, stream=None):
    """w13 [E, 2I, H] (gate rows then up rows), w2 [E, H, I], bf16 CUDA."""
    E, I2, H = w13.shape
    I = I2 // 2
    assert w2.shape == (E, H, I)
    L = lib()
    dev = w13.device
    q13 = empty_qtensor(NVFP4, E * 2 * I, H, dev, n_global=E)
    q2 = empty_qtensor(NVFP4, E * H, I, dev, n_global=E)
    ws = _ws(L.fp4_moe_prepack_workspace_size(E, H, I), dev)
    _check(L.fp4_moe_prepack_weights(_ptr(w13), _ptr(w2), E, H, I, _ptr(q13.codes), _ptr(q13.scales),
                                     _ptr(q13.gscale), _ptr(q2.codes), _ptr(q2.scales), _ptr(q2.gscale), _ptr(ws),
                                     ws.numel(), _stream(stream)))
    return MoEWeights(E, H, I, q13, q2)


def _host_scales(a, E):
    if a is None:
        return None
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float32).reshape(-1))
    assert arr.size == E
    return arr


MOE_AUTO, MOE_CHAIN, MOE_FUSED = 0, 1, 2


def set_moe_policy(policy):
    """Choose the MoE implementation (MOE_AUTO: one launch for a few tokens;
    MOE_CHAIN; MOE_FUSED: one launch wherever its shapes apply)."""
    _check(lib().fp4_set_moe_policy(int(policy)))


def moe_workspace_layout(T, H, I, E, top_k):
    L = lib()
    offs = (ctypes.c_int64 * 32)()
    n = L.fp4_moe_workspace_layout(T, H, I, E, top_k, offs, 32)
    return [offs[i] for i in range(n)]


def moe(hidden, logits, mw, top_k, mode=DYNAMIC, static13=None, static2=None, out=None, workspace=None,
        stage_mask=None, stream=None):
    """NVFP4 fused MoE forward: hidden bf16 [T, H], logits fp32 [T, E]."""
    T, H = hidden.shape
    E = logits.shape[1]
    L = lib()
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=hidden.device)
    wsb = L.fp4_moe_workspace_size(T, H, mw.I, E, top_k)
    ws = workspace if workspace is not None else _ws(wsb, hidden.device)
    s13 = _host_scales(static13, E)
    s2 = _host_scales(static2, E)
    p13 = _P(0) if s13 is None else _P(s13.ctypes.data)
    p2 = _P(0) if s2 is None else _P(s2.ctypes.data)
    args = [_ptr(hidden), _ptr(logits), T, H, mw.I, E, top_k, mode, p13, p2, _ptr(mw.w13.codes),
            _ptr(mw.w13.scales), _ptr(mw.w13.gscale), _ptr(mw.w2.codes), _ptr(mw.w2.scales), _ptr(mw.w2.gscale),
            _ptr(out), _ptr(ws), ws.numel()]
    if stage_mask is None:
        _check(L.fp4_moe_grouped(*args, _stream(stream)))
    else:
        _check(L.fp4_moe_grouped_stages(*args, stage_mask, _stream(stream)))
    return out
