"""Pins of the MXFP8 / MXFP6 oracle (``oracle/mx_wide.py``) against things
other than itself: torch's float8 conversions (library routines), the value
sets written out from the formats' definitions, an exact-rational brute force
of the rounding, and the MXFP4 quantiser written independently in C."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from mxfp4_block_scaled_gb300 import inputs as I
from oracle import mx_wide as X

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_decode_matches_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    got = X.decode(fmt, codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_encode_matches_torch(fmt):
    """Round to nearest even inside the finite range, against torch's fp32 ->
    float8 conversion, on random magnitudes and on every exact midpoint."""
    rng = np.random.default_rng(3)
    top = X.max_finite(fmt)
    v = rng.standard_normal(20000) * np.exp2(rng.integers(-20, 16, 20000))
    v = v[np.abs(v) <= top]
    _, g = X.grid(fmt)
    mids = (g[1:] + g[:-1]) / 2
    v = np.concatenate([v, mids, -mids, g, -g]).astype(np.float32)
    want = torch.from_numpy(v).to(TORCH_FP8[fmt]).view(torch.uint8).numpy().astype(np.int64)
    got = X.encode(fmt, v.astype(np.float64))
    assert np.array_equal(got, want)


def test_fp6_value_sets_from_their_definitions():
    """E2M3: subnormals m/8 (m < 8), normals (1 + m/8) 2^(e-1) for e = 1..3.
    E3M2: subnormals m/16 (m < 4), normals (1 + m/4) 2^(e-3) for e = 1..7."""
    e2m3 = {Fraction(m, 8) for m in range(8)} | {(1 + Fraction(m, 8)) * Fraction(2) ** (e - 1)
                                                  for e in range(1, 4) for m in range(8)}
    e3m2 = {Fraction(m, 16) for m in range(4)} | {(1 + Fraction(m, 4)) * Fraction(2) ** (e - 3)
                                                   for e in range(1, 8) for m in range(4)}
    for fmt, want in (("e2m3", e2m3), ("e3m2", e3m2)):
        codes, vals = X.grid(fmt)
        assert len(codes) == 32 and {Fraction(float(v)) for v in vals} == want
        assert list(codes) == list(range(32))  # every 6-bit pattern is a finite value
    assert X.max_finite("e2m3") == 7.5 and X.max_finite("e3m2") == 28.0
    assert X.max_finite("e4m3") == 448.0 and X.max_finite("e5m2") == 57344.0


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e3m2", "e4m3", "e5m2"])
def test_encode_against_exact_brute_force(fmt):
    """Nearest grid value in exact rationals, ties to the even code, values
    beyond the top saturate, the sign is kept (also for zero)."""
    codes, vals = X.grid(fmt)
    grid = [(Fraction(float(v)), int(c)) for c, v in zip(codes, vals)]
    rng = np.random.default_rng(11)
    top = float(vals[-1])
    v = np.concatenate([rng.uniform(-1.2 * top, 1.2 * top, 300), rng.uniform(-1, 1, 100) * float(vals[2]),
                        (vals[1:] + vals[:-1]) / 2, [0.0, -0.0, top, -top, 2 * top]])
    got = X.encode(fmt, v)
    sbit = 1 << (X.code_bits(fmt) - 1)
    for x, g in zip(v, got):
        a = abs(Fraction(float(x)))
        best = min(grid, key=lambda p: (abs(p[0] - a), p[1] % 2))  # nearest, then the even code
        if a >= grid[-1][0]:
            best = grid[-1]
        want = best[1] | (sbit if np.signbit(x) else 0)
        assert int(g) == want, (fmt, x, int(g), want)


def test_generic_rule_reproduces_the_c_mxfp4_quantiser(O):
    """With E2M1 elements the generic MX rule must give the MXFP4 oracle's
    codes and scales bit for bit (two independent implementations)."""
    x = I.activations_with_outliers(8, 1024, 5)
    u = I.u16(x).copy()
    u[0, :32] = 0                      # an all-zero block
    u[1, 32:64] = 0x8000               # a block of negative zeros
    u[2, :32] = np.uint16(0x3F80)      # all 1.0: amax an exact power of two
    c_codes, c_scales = O.quantize_mxfp4(u)
    g_codes, g_scales = X.quantize("e2m1", u)
    packed = (g_codes[:, 0::2] | (g_codes[:, 1::2] << 4)).astype(np.uint8)
    assert np.array_equal(g_scales, c_scales)
    assert np.array_equal(packed, c_codes)


@pytest.mark.parametrize("fmt", ["e2m3", "e3m2", "e4m3", "e5m2"])
def test_scale_rule_invariants(fmt):
    rng = np.random.default_rng(5)
    x = torch.from_numpy((rng.standard_normal((16, 256)) * np.exp2(rng.integers(-30, 30, (16, 1))))
                         .astype(np.float32)).to(torch.bfloat16)
    u = I.u16(x).copy()
    u[3, 64:96] = 0
    codes, scales = X.quantize(fmt, u)
    xf = X.bf16_to_f64(u).reshape(16, 8, 32)
    amax = np.abs(xf).max(axis=2)
    emax = X.FORMATS[fmt][3]
    nz = amax > 0
    # the scaled block maximum lies in [2^emax, 2^(emax+1))
    sc = np.ldexp(amax[nz], -(scales[nz].astype(np.int32) - 127))
    assert ((sc >= 2.0 ** emax) & (sc < 2.0 ** (emax + 1))).all()
    assert (scales[~nz] == 0).all() and (codes.reshape(16, 8, 32)[~nz] == 0).all()
    # dequantised values are within half a grid step (relative to the block scale) of the input,
    # except where they saturate at the top value
    d = X.dequantize(fmt, codes, scales).reshape(16, 8, 32)
    top = X.max_finite(fmt) * np.ldexp(1.0, scales.astype(np.int32) - 127)[..., None]
    rel = X.FORMATS[fmt][1]
    err_ok = np.abs(d - xf) <= np.maximum(np.abs(xf) * 2.0 ** -(rel + 1),
                                          np.ldexp(1.0, scales.astype(np.int32) - 127 + 1 - X.FORMATS[fmt][2]
                                                   - rel)[..., None] / 2 + 1e-300)
    assert (err_ok | (np.abs(xf) >= top)).all()


@pytest.mark.parametrize("fmt", ["e2m3", "e4m3", "e5m2"])
def test_mx_wide_gemm_exact_on_tiny_shapes(fmt):
    """gemm = exact rational sum of the hand-decoded operands (fp64 result
    within its own rounding)."""
    a = I.randn_bf16((2, 64), 21)
    w = I.randn_bf16((3, 64), 22, std=0.02)
    ca, sa = X.quantize(fmt, I.u16(a))
    cb, sb = X.quantize(fmt, I.u16(w))
    out, _ = X.gemm(fmt, ca, sa, fmt, cb, sb)
    for i in range(2):
        for j in range(3):
            s = Fraction(0)
            for k in range(64):
                va = Fraction(float(X.decode(fmt, ca[i, k]))) * Fraction(2) ** (int(sa[i, k // 32]) - 127)
                vb = Fraction(float(X.decode(fmt, cb[j, k]))) * Fraction(2) ** (int(sb[j, k // 32]) - 127)
                s += va * vb
            assert abs(Fraction(out[i, j]) - s) <= abs(s) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 300)


@pytest.mark.parametrize("fmt,bound", [("e4m3", 0.05), ("e5m2", 0.1), ("e2m3", 0.05), ("e3m2", 0.1)])
def test_mx_wide_linear_close_to_the_unquantised_product(fmt, bound):
    """A wrong scale (a factor of two anywhere) or a transposed operand fails this."""
    a = I.randn_bf16((32, 256), 31)
    w = I.randn_bf16((48, 256), 32, std=0.02)
    out, _ = X.linear(fmt, I.u16(a), I.u16(w))
    ref = a.double().numpy() @ w.double().numpy().T
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < bound
