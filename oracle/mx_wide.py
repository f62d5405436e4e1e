"""CPU oracle for the wider MX formats: MXFP8 (E4M3, E5M2 elements) and
MXFP6 (E2M3, E3M2 elements), 32-element blocks with one E8M0 scale.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/`` may
import it, and it shares no code with the CUDA library.

Source: "vLLM per-format kernel capability matrix" lists MXFP4, MXFP6 and
MXFP8 with group size 32 (the record header on group sizes).  The pages do
not define the element formats or the scale rule for FP6/FP8, so this module
takes the plainest reading.  It is the rule the pages give for MXFP4 ("vLLM
on DGX Spark: technical report", section 6.4), with the element's own
largest exponent in place of E2M1's:
  - element formats: sign, E exponent bits with bias b, M mantissa bits,
    subnormals at exponent field 0; E4M3 has no infinities and one NaN
    pattern per sign (S.1111.111), E5M2 has IEEE infinities and NaNs, and
    E2M3 / E3M2 have neither;
  - shared exponent e = floor(log2 amax_b) - emax, where emax is the
    exponent of the element's largest normal (E4M3 8, E5M2 15, E2M3 2,
    E3M2 4, E2M1 2), clamped to [-127, 127] and stored as the byte e + 127;
  - elements: x / 2^e (exact), rounded to nearest with ties to the even
    code, saturating at the largest finite value; the sign of a value that
    rounds to zero is kept; an all-zero block gets scale byte 0 and code 0.
E2M1 is included as a format so that the generic rule can be checked against
the MXFP4 quantiser written independently in ``fp4_oracle.c``.

All arithmetic is in fp64 on exact values: bf16 inputs, power-of-two scales
and the format grids are all exact in fp64, so the only rounding is the
element rounding itself, done by choosing from the enumerated grid.
"""
import numpy as np

# name -> (exponent bits, mantissa bits, bias, emax, has_inf_nan, e4m3_style_nan)
FORMATS = {
    "e2m1": (2, 1, 1, 2, False, False),
    "e2m3": (2, 3, 1, 2, False, False),
    "e3m2": (3, 2, 3, 4, False, False),
    "e4m3": (4, 3, 7, 8, False, True),
    "e5m2": (5, 2, 15, 15, True, False),
}
BLOCK = 32


def code_bits(fmt):
    e, m = FORMATS[fmt][:2]
    return 1 + e + m


def decode(fmt, codes):
    """Element codes (integers) -> values (fp64), from the bit fields; NaN /
    inf where the format defines them."""
    E, M, bias, _, ieee, e4m3 = FORMATS[fmt]
    c = np.asarray(codes, dtype=np.int64)
    sign = (c >> (E + M)) & 1
    ef = (c >> M) & ((1 << E) - 1)
    mf = c & ((1 << M) - 1)
    sub = np.ldexp(mf.astype(np.float64), 1 - bias - M)  # 0.m x 2^(1-bias)
    nrm = np.ldexp((mf + (1 << M)).astype(np.float64), (ef - bias - M).astype(np.int32))  # 1.m x 2^(e-bias)
    v = np.where(ef == 0, sub, nrm)
    emax_field = (1 << E) - 1
    if ieee:
        v = np.where(ef == emax_field, np.where(mf == 0, np.inf, np.nan), v)
    if e4m3:
        v = np.where((ef == emax_field) & (mf == (1 << M) - 1), np.nan, v)
    return np.where(sign == 1, -v, v)


def grid(fmt):
    """(codes, values) of the finite non-negative values, ascending."""
    n = 1 << (code_bits(fmt) - 1)
    codes = np.arange(n, dtype=np.int64)
    vals = decode(fmt, codes)
    ok = np.isfinite(vals)
    return codes[ok], vals[ok]


def max_finite(fmt):
    return grid(fmt)[1][-1]


def encode(fmt, v):
    """fp64 values -> codes: nearest grid value, ties to the even code,
    saturating at the largest finite value; the sign bit follows the input's
    sign (also for results that round to zero)."""
    v = np.asarray(v, dtype=np.float64)
    gc, gv = grid(fmt)
    a = np.abs(v)
    hi = np.searchsorted(gv, a, side="left")  # gv[hi - 1] < a <= gv[hi]
    hi_c = np.minimum(hi, len(gv) - 1)
    lo_c = np.maximum(hi - 1, 0)
    d_hi = gv[hi_c] - a
    d_lo = a - gv[lo_c]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (gc[hi_c] % 2 == 0))
    mag = np.where(pick_hi, gc[hi_c], gc[lo_c])
    mag = np.where(a >= gv[-1], gc[-1], mag)  # saturate (also at and beyond the top value)
    mag = np.where(a == 0, 0, mag)
    sign = np.signbit(v).astype(np.int64) << (code_bits(fmt) - 1)
    return (mag | sign).astype(np.int64)


def bf16_to_f64(u16):
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def quantize(fmt, x_u16):
    """x: [rows, k] bf16 bits, k % 32 == 0 -> (codes [rows, k] int64, one per
    element; scales [rows, k/32] uint8 E8M0)."""
    x = bf16_to_f64(x_u16)
    rows, k = x.shape
    assert k % BLOCK == 0
    xb = x.reshape(rows, k // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=2)
    _, ex = np.frexp(amax)  # amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1
    e = np.clip(ex - 1 - FORMATS[fmt][3], -127, 127).astype(np.int32)
    nz = amax > 0
    scales = np.where(nz, e + 127, 0).astype(np.uint8)
    q = np.ldexp(xb, -e[..., None])
    codes = np.where(nz[..., None], encode(fmt, q), 0)
    return codes.reshape(rows, k), scales


def dequantize(fmt, codes, scales):
    """codes [rows, k], scales [rows, k/32] -> fp64 values (element x 2^(byte - 127))."""
    codes = np.asarray(codes)
    rows, k = codes.shape
    s = np.ldexp(1.0, np.asarray(scales, dtype=np.int32) - 127)
    return (decode(fmt, codes).reshape(rows, k // BLOCK, BLOCK) * s[..., None]).reshape(rows, k)


def gemm(fmt_a, ca, sa, fmt_b, cb, sb):
    """Dequantise both operands, then fp64: out [m, n] = A . B^T, and the
    magnitude sum sum_k |A||B| that sizes an fp32 accumulation bound."""
    da = dequantize(fmt_a, ca, sa)
    db = dequantize(fmt_b, cb, sb)
    return da @ db.T, np.abs(da) @ np.abs(db).T


def linear(fmt, x_u16, w_u16):
    """Both operands quantised to `fmt` by `quantize`, then `gemm`."""
    ca, sa = quantize(fmt, x_u16)
    cb, sb = quantize(fmt, w_u16)
    return gemm(fmt, ca, sa, fmt, cb, sb)
