"""Pins of the CPU oracle against facts that do not come from the oracle
itself: the printed value set, hand-derived worked blocks, closed forms,
library conversions (torch's float8_e4m3fn / bf16), exact rational brute force
and invariants.  CPU only."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden
from mxfp4_block_scaled_gb300 import inputs as I


def _bf16_bits(vals):
    return I.u16(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


# --------------------------------------------------------------- E2M1 codec

def test_e2m1_value_set_matches_golden(O):
    _, rows = read_golden("e2m1_values.txt")
    for code, val in rows:
        got = O.e2m1_decode(int(code))
        want = float(val)
        assert got == want and math.copysign(1, got) == math.copysign(1, want), (code, got, want)


def test_e2m1_closed_form_from_bits(O):
    # 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = (m / 2.0) if e == 0 else (2.0 ** (e - 1)) * (1 + m / 2.0)
        assert O.e2m1_decode(code) == (-mag if s else mag)


def test_e2m1_round_trip_all_codes(O):
    for code in range(16):
        assert O.e2m1_encode(O.e2m1_decode(code)) == code


def _nearest_even_on_grid(v, grid):
    """Brute force: nearest grid magnitude, ties to the even index."""
    a = abs(v)
    best = min(range(len(grid)), key=lambda i: (abs(a - grid[i]), i & 1))
    return best


def test_e2m1_brute_force_random(O):
    grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.uniform(-7, 7, 4000), rng.uniform(-0.3, 0.3, 500)]).astype(np.float32)
    for v in vals:
        v = float(v)
        c = O.e2m1_encode(v)
        want = _nearest_even_on_grid(v, grid) if abs(v) < 6 else 7
        assert (c & 7) == want, (v, c)
        assert (c >> 3) == (1 if math.copysign(1, v) < 0 else 0)


def test_e2m1_ties_and_neighbours(O):
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for mid, code in ties.items():
        assert O.e2m1_encode(mid) == code
        assert O.e2m1_encode(-mid) == code | 8
        up = float(np.nextafter(np.float32(mid), np.float32(np.inf)))
        dn = float(np.nextafter(np.float32(mid), np.float32(-np.inf)))
        grid = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
        lo = max(i for i in range(8) if grid[i] < mid)
        assert O.e2m1_encode(up) == lo + 1
        assert O.e2m1_encode(dn) == lo


def test_e2m1_saturation(O):
    for v in [6.0, 6.5, 7.99, 100.0, 1e30, float("inf")]:
        assert O.e2m1_encode(v) == 7
        assert O.e2m1_encode(-v) == 15


# --------------------------------------------------------------- E4M3 codec

def test_e4m3_decode_matches_torch(O):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = O.e4m3_decode(b)
        if np.isnan(ref[b]):
            assert math.isnan(got)
        else:
            assert got == ref[b], (b, got, ref[b])
    assert O.e4m3_decode(0x7E) == 448.0 and O.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range(O):
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(0, 448, 3000), np.exp(rng.uniform(np.log(1e-4), np.log(448), 3000)),
                           rng.uniform(0, 2.0 ** -6, 1000)]).astype(np.float32)
    # every midpoint between consecutive finite codes and its neighbours
    mags = [O.e4m3_decode(b) for b in range(0x7F)]
    mids = [(mags[i] + mags[i + 1]) / 2 for i in range(len(mags) - 1)]
    extra = []
    for m in mids:
        m32 = np.float32(m)
        extra += [m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0))]
    vals = np.concatenate([vals, np.array(extra, dtype=np.float32)])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_encode(float(v)) for v in vals], dtype=np.uint8)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), got[i], ref[i]) for i in bad[:10]]


def test_e4m3_round_trip_and_saturation(O):
    for b in range(0x7F):
        assert O.e4m3_encode(O.e4m3_decode(b)) == b
    for v in [448.0, 449.0, 464.0, 500.0, 1e20, float("inf")]:
        assert O.e4m3_encode(v) == 0x7E
    assert O.e4m3_encode(2.0 ** -10) == 0          # tie between 0 and 2^-9 -> even (0)
    assert O.e4m3_encode(1.5 * 2.0 ** -9) == 2      # tie between 1 and 2 (x 2^-9) -> even


# --------------------------------------------------------------- E8M0, bf16

def test_e8m0_all_exponents(O):
    for b in range(255):
        assert O.e8m0_decode(b) == math.ldexp(1.0, b - 127)
    assert math.isnan(O.e8m0_decode(255))


def test_bf16_conversions_match_torch(O):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f32_to_bf16(x)
    assert np.array_equal(got, ref)
    assert np.array_equal(O.bf16_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())
    # fp64 -> bf16 in one rounding: compare with exact rational nearest
    vals = np.concatenate([rng.standard_normal(300) * 1e-3, rng.standard_normal(300) * 1e3])
    for v in vals:
        b0 = int(np.float32(v).view(np.uint32) >> 16)
        cands = list(range(b0 - 2, b0 + 3))
        cvals = [Fraction(float(O.bf16_to_f32(np.array([b], dtype=np.uint16))[0])) for b in cands]
        best = min(range(len(cands)), key=lambda i: (abs(cvals[i] - Fraction(float(v))), cands[i] & 1))
        assert Fraction(float(O.bf16_round(v))) == cvals[best]


# ------------------------------------------------------------- scale layout

@pytest.mark.parametrize("rows,k,fmt", [(1, 32, 1), (130, 512, 0), (256, 4096, 0), (300, 800, 1), (128, 16, 0)])
def test_scale_layout_is_bijection(O, rows, k, fmt):
    blk = O.BLOCK[fmt]
    ksf_pad = O.scale_cols_padded(k, fmt)
    rows_pad = (rows + 127) // 128 * 128
    total = O.scale_mma_bytes(rows, k, fmt)
    assert total == rows_pad * ksf_pad and ksf_pad % (256 // blk) == 0 and ksf_pad * blk >= k
    idx = np.array([[O.scale_mma_index(r, j, ksf_pad) for j in range(ksf_pad)] for r in range(rows_pad)])
    assert np.array_equal(np.sort(idx.ravel()), np.arange(total))
    canon = np.random.default_rng(1).integers(0, 256, (rows, k // blk), dtype=np.uint8)
    mma = O.scales_to_mma(canon, rows, k, fmt)
    assert np.array_equal(O.scales_from_mma(mma, rows, k, fmt), canon)
    pad = np.ones(total, bool)
    pad[idx[:rows, :k // blk].ravel()] = False
    assert np.all(mma[pad] == 0)


def test_scale_layout_fixed_points(O):
    # 512-byte atoms of 128 rows x 4 scale columns; row r at (r%32)*16 + (r//32)*4
    ksf = 16
    assert O.scale_mma_index(0, 0, ksf) == 0
    assert O.scale_mma_index(1, 0, ksf) == 16
    assert O.scale_mma_index(32, 0, ksf) == 4
    assert O.scale_mma_index(0, 3, ksf) == 3
    assert O.scale_mma_index(0, 4, ksf) == 512
    assert O.scale_mma_index(127, 15, ksf) == 3 * 512 + 31 * 16 + 3 * 4 + 3
    assert O.scale_mma_index(128, 0, ksf) == 4 * 512


# -------------------------------------------------------- worked examples

def _golden_case(name):
    kv, _ = read_golden(name)
    x = np.array([float(v) for v in kv["x"]], dtype=np.float32)
    scales = np.array([int(v, 16) for v in kv["scales"]], dtype=np.uint8)
    codes = np.array([int(v, 16) for v in kv["codes"]], dtype=np.uint8)
    return x, scales, codes


def test_nvfp4_worked_blocks(O):
    x, scales, codes = _golden_case("nvfp4_worked_blocks.txt")
    xb = _bf16_bits(x).reshape(1, -1)
    assert np.array_equal(O.bf16_to_f32(xb).ravel(), x)      # fixture values are bf16-exact
    c, s, sg = O.quantize_nvfp4(xb, O.STATIC, 1.0)
    assert sg == 1.0
    assert np.array_equal(s.ravel(), scales), s
    assert np.array_equal(c.ravel(), codes), [hex(v) for v in c.ravel()]


def test_mxfp4_worked_blocks(O):
    x, scales, codes = _golden_case("mxfp4_worked_blocks.txt")
    xb = _bf16_bits(x).reshape(1, -1)
    c, s = O.quantize_mxfp4(xb)
    assert np.array_equal(s.ravel(), scales), s
    assert np.array_equal(c.ravel(), codes), [hex(v) for v in c.ravel()]


# ---------------------------------------------------- quantiser invariants

def _grid_halfstep(v):
    """Half the spacing of the E2M1 grid interval containing |v| (v <= 6)."""
    a = abs(v)
    return 0.25 if a <= 2 else (0.5 if a <= 4 else 1.0)


def test_nvfp4_dynamic_invariants(O):
    x = I.randn_bf16((8, 256), 11)
    x[3, 37] = 9.5  # the tensor amax
    xb = I.u16(x)
    xf = O.bf16_to_f32(xb).reshape(8, 256).astype(np.float64)
    c, s, sg = O.quantize_nvfp4(xb)
    amax = np.abs(xf).max()
    assert sg == np.float32(np.float32(amax) / np.float32(2688.0))
    assert s[3, 37 // 16] == 0x7E  # block holding the amax gets the largest scale, 448
    deq = O.dequantize(O.NVFP4, c, s, sg)
    d = np.repeat(O.e4m3_table()[s] * sg, 16, axis=1)
    err = np.abs(deq - xf)
    ratio = xf / d
    ok = np.abs(ratio) <= 6
    # a correctly rounded element is within half a grid step of x (tiny slack for fp32 x/d)
    half = np.vectorize(_grid_halfstep)(ratio) * d
    assert np.all(err[ok] <= half[ok] * (1 + 1e-6) + 1e-30)
    assert np.all(np.abs(deq) <= 6 * d + 1e-30)


def test_nvfp4_zero_tensor_and_zero_block(O):
    z = np.zeros((2, 64), dtype=np.uint16)
    c, s, sg = O.quantize_nvfp4(z)
    assert sg == 0.0 and not c.any() and not s.any()
    x = I.randn_bf16((1, 64), 2)
    x[0, 16:32] = 0
    c, s, sg = O.quantize_nvfp4(I.u16(x))
    assert s[0, 1] == 0 and not c[0, 8:16].any() and s[0, 0] != 0


def test_nvfp4_block_locality(O):
    x = I.randn_bf16((1, 64), 4)
    x[0, 0] = 5.0  # keep the tensor amax fixed
    c0, s0, g0 = O.quantize_nvfp4(I.u16(x))
    y = x.clone()
    y[0, 40] = y[0, 40] * 0.5
    c1, s1, g1 = O.quantize_nvfp4(I.u16(y))
    assert g0 == g1
    assert np.array_equal(c0[0, :16], c1[0, :16]) and np.array_equal(c0[0, 24:], c1[0, 24:])
    assert np.array_equal(s0[0, [0, 1, 3]], s1[0, [0, 1, 3]])


def test_nvfp4_static_exact_round_trip(O):
    # values on the E2M1 grid times 2 with a block amax of 12: scale 2.0 exactly
    rng = np.random.default_rng(8)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6], dtype=np.float32)
    x = rng.choice(grid, (4, 64)) * 2
    x[:, ::16] = 12.0
    xb = _bf16_bits(x.ravel()).reshape(4, 64)
    c, s, _ = O.quantize_nvfp4(xb, O.STATIC, 1.0)
    assert np.all(s == 0x40)
    assert np.array_equal(O.dequantize(O.NVFP4, c, s, 1.0), x.astype(np.float64))


def test_nvfp4_static_saturates(O):
    x = np.array([1000.0] + [1.0] * 15, dtype=np.float32)
    c, s, sg = O.quantize_nvfp4(_bf16_bits(x).reshape(1, 16), O.STATIC, 0.01)
    assert s[0, 0] == 0x7E and (c[0, 0] & 15) == 7   # 448 and 6: both clamp


def test_mxfp4_scale_rule_and_round_trip(O):
    rng = np.random.default_rng(9)
    x = I.randn_bf16((16, 256), 21)
    xb = I.u16(x)
    xf = O.bf16_to_f32(xb).reshape(16, 256)
    c, s = O.quantize_mxfp4(xb)
    for r in range(16):
        for b in range(8):
            amax = float(np.abs(xf[r, b * 32:(b + 1) * 32]).max())
            e = math.frexp(amax)[1] - 1 - 2
            assert s[r, b] == e + 127
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -6, -4], dtype=np.float32)
    y = rng.choice(grid, (2, 64)) * np.float32(2.0 ** -5)
    y[:, 0] = 6 * 2.0 ** -5
    y[:, 32] = -6 * 2.0 ** -5
    c2, s2 = O.quantize_mxfp4(_bf16_bits(y.ravel()).reshape(2, 64))
    assert np.all(s2 == 127 - 5)
    assert np.array_equal(O.dequantize(O.MXFP4, c2, s2), y.astype(np.float64))


# --------------------------------------------------------------------- GEMM

def _exact_gemm_fraction(fmt, ca, sa, cb, sb):
    """Exact rational S[m][n] = sum_k deqA * deqB from the raw bits, with the
    E2M1 / E4M3 / E8M0 values re-derived here from their bit definitions."""
    def e2m1(c):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
        return -mag if s else mag

    def e4m3(b):
        e, m = (b >> 3) & 15, b & 7
        return Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)

    def e8m0(b):
        return Fraction(2) ** (b - 127)

    blk = 16 if fmt == 0 else 32
    dec = e4m3 if fmt == 0 else e8m0
    M, N, K = ca.shape[0], cb.shape[0], ca.shape[1] * 2

    def val(codes, scales, r, k):
        byte = int(codes[r, k // 2])
        c = (byte >> 4) if (k & 1) else (byte & 15)
        return e2m1(c) * dec(int(scales[r, k // blk]))

    return [[sum(val(ca, sa, m, k) * val(cb, sb, n, k) for k in range(K)) for n in range(N)] for m in range(M)]


@pytest.mark.parametrize("fmt,M,N,K", [(0, 3, 4, 16), (0, 2, 3, 64), (1, 4, 2, 32), (1, 3, 3, 64)])
def test_gemm_brute_force_tiny(O, fmt, M, N, K):
    a = I.randn_bf16((M, K), 31 + K)
    w = I.randn_bf16((N, K), 41 + K, std=0.02)
    out, mag, qa, qw = O.linear(fmt, I.u16(a), I.u16(w))
    S = _exact_gemm_fraction(fmt, qa[0], qa[1], qw[0], qw[1])
    alpha = Fraction(O.alpha_of(fmt, qa[2], qw[2]))
    for m in range(M):
        for n in range(N):
            want = alpha * S[m][n]
            assert abs(Fraction(out[m, n]) - want) <= abs(want) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)
    if fmt == 0:
        S20 = O.gemm_nvfp4_exact(qa[0], qa[1], qw[0], qw[1])
        for m in range(M):
            for n in range(N):
                assert Fraction(int(S20[m, n]), 2 ** 20) == S[m][n]


def test_gemm_exact_int_path_agrees_with_fp64(O):
    a = I.randn_bf16((9, 512), 51)
    w = I.randn_bf16((7, 512), 52, std=0.02)
    out, mag, qa, qw = O.linear(O.NVFP4, I.u16(a), I.u16(w))
    S20 = O.gemm_nvfp4_exact(qa[0], qa[1], qw[0], qw[1])
    alpha = O.alpha_of(O.NVFP4, qa[2], qw[2])
    exact = alpha * S20.astype(np.float64) / 2 ** 20
    assert np.all(np.abs(exact - out) <= 1e-14 * mag)


def test_gemm_transpose_symmetry(O):
    a = I.randn_bf16((5, 256), 61)
    w = I.randn_bf16((6, 256), 62)
    qa = O.quantize_nvfp4(I.u16(a))
    qw = O.quantize_nvfp4(I.u16(w))
    o1, _ = O.gemm(O.NVFP4, *qa, *qw)
    o2, _ = O.gemm(O.NVFP4, *qw, *qa)
    assert np.allclose(o1, o2.T, rtol=1e-15, atol=0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_linear_close_to_unquantised_matmul(O, fmt):
    # catches a wrong alpha / scale convention: W4A4 error is ~10%, not O(1)
    a = I.randn_bf16((32, 1024), 71)
    w = I.randn_bf16((64, 1024), 72, std=0.02)
    out, _, _, _ = O.linear(fmt, I.u16(a), I.u16(w))
    ref = a.double().numpy() @ w.double().numpy().T
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert 0.01 < rel < 0.2, rel


# ------------------------------------------------------------- W4A16 linear

@pytest.mark.parametrize("fmt,M,N,K", [(0, 2, 3, 32), (1, 3, 2, 64)])
def test_w4a16_brute_force_tiny(O, fmt, M, N, K):
    """Exact rational sum of x times the hand-decoded weights."""
    x = I.randn_bf16((M, K), 81 + K)
    w = I.randn_bf16((N, K), 82 + K, std=0.02)
    cw, sw, gw = O.quantize(fmt, I.u16(w))
    out, _ = O.linear_w4a16(fmt, I.u16(x), cw, sw, gw)
    e2m1 = lambda c: (-1) ** (c >> 3) * [0, 0.5, 1, 1.5, 2, 3, 4, 6][c & 7]
    blk = 16 if fmt == 0 else 32
    dec = (lambda b: Fraction(O.e4m3_decode(b))) if fmt == 0 else (lambda b: Fraction(2) ** (b - 127))
    g = Fraction(1) if fmt == 1 else Fraction(float(np.float32(gw)))
    xf = x.float().numpy()
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                byte = int(cw[n, k // 2])
                c = (byte >> 4) if (k & 1) else (byte & 15)
                s += Fraction(float(xf[m, k])) * Fraction(e2m1(c)) * dec(int(sw[n, k // blk]))
            want = g * s
            assert abs(Fraction(out[m, n]) - want) <= abs(want) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_w4a16_one_hot_reads_the_weights(O):
    """x = e_k selects column k of the dequantised weights, times s_gW."""
    K, N = 256, 8
    w = I.randn_bf16((N, K), 91, std=0.02)
    cw, sw, gw = O.quantize_nvfp4(I.u16(w))
    dw = O.dequantize(O.NVFP4, cw, sw, gw)
    for k in (0, 17, 128, 255):
        x = torch.zeros((1, K), dtype=torch.bfloat16)
        x[0, k] = 1.0
        out, _ = O.linear_w4a16(O.NVFP4, I.u16(x), cw, sw, gw)
        assert np.array_equal(out[0], dw[:, k])


@pytest.mark.parametrize("fmt", [0, 1])
def test_w4a16_equals_w4a4_on_fp4_exact_activations(O, fmt):
    """Activations whose quantisation is exact (FP4 values times a power-of-two
    block scale) give the same output through the W4A4 oracle."""
    rng = np.random.default_rng(7)
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    M, K, N = 4, 256, 6
    a = rng.choice(vals, size=(M, K)) * rng.choice([-1, 1], size=(M, K))
    a[:, ::16] = 6.0  # every 16-block holds the largest value
    x = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    w = I.randn_bf16((N, K), 93, std=0.02)
    cw, sw, gw = O.quantize(fmt, I.u16(w))
    out16, _ = O.linear_w4a16(fmt, I.u16(x), cw, sw, gw)
    if fmt == 0:
        # with s_g = 2^-8 every block's scale byte is E4M3(6 / (6 * 2^-8)) = 256,
        # so the divisor 256 * 2^-8 is exactly 1 and the codes are exact
        ca, sa, ga = O.quantize_nvfp4(I.u16(x), O.STATIC, 1.0 / 256.0)
    else:
        ca, sa = O.quantize_mxfp4(I.u16(x))
        ga = 1.0
    deq = O.dequantize(fmt, ca, sa, ga)
    assert np.array_equal(deq, a.astype(np.float64))  # the activations' quantisation is exact
    out4, _ = O.gemm(fmt, ca, sa, ga, cw, sw, gw)
    assert np.allclose(out16, out4, rtol=1e-14, atol=0)


# ----------------------------------------------------------- router/permute

def test_router_invariants_and_brute_force(O):
    T, E, k = 50, 128, 8
    logits = I.router_logits(T, E, 5).numpy()
    ids, w = O.router_topk(logits, k)
    for t in range(T):
        assert len(set(ids[t].tolist())) == k and np.all((ids[t] >= 0) & (ids[t] < E))
        assert np.all(w[t] > 0) and abs(w[t].sum() - 1) < 1e-12 and np.all(np.diff(w[t]) <= 0)
        # independent: full softmax in fp64, Python sort by (-p, index), renormalise
        z = np.exp(logits[t].astype(np.float64) - logits[t].max())
        p = z / z.sum()
        top = sorted(range(E), key=lambda i: (-p[i], i))[:k]
        assert ids[t].tolist() == top
        assert np.allclose(w[t], p[top] / p[top].sum(), rtol=1e-12)


def test_router_ties_go_to_lower_index(O):
    logits = np.zeros((2, 16), dtype=np.float32)
    logits[0, [3, 9, 12]] = 1.0
    ids, w = O.router_topk(logits, 4)
    assert ids[0].tolist() == [3, 9, 12, 0]
    assert ids[1].tolist() == [0, 1, 2, 3] and np.allclose(w[1], 0.25)


def test_permute_against_loop(O):
    rng = np.random.default_rng(0)
    T, k, E = 40, 4, 16
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, order = O.permute(ids, E)
    want = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    want.append(t * k + j)
    assert order.tolist() == want
    assert counts.sum() == T * k and offsets[0] == 0 and np.all(np.diff(offsets) == counts)


# ---------------------------------------------------------------------- MoE

def test_silu_closed_form(O):
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(40.0) - 40.0) < 1e-12
    g = np.linspace(-8, 8, 33)
    assert np.allclose(O.silu(-g), O.silu(g) - g, atol=1e-14)
    assert np.allclose(O.silu(g), g * (1 / (1 + np.exp(-g))))


def _small_moe(T=6, E=4, H=64, Inter=32, k=2, seed=0):
    hidden = I.randn_bf16((T, H), seed + 1)
    logits = I.router_logits(T, E, seed + 2).numpy()
    w13 = I.expert_weights_bf16(E, 2 * Inter, H, seed + 3, std=0.1)
    w2 = I.expert_weights_bf16(E, H, Inter, seed + 4, std=0.1)
    return hidden, logits, w13, w2


def test_moe_per_token_loop(O):
    """The batched sort/permute/unpermute oracle equals a per-token loop over
    each token's experts (the requantisation scale of h is per expert)."""
    hidden, logits, w13, w2 = _small_moe()
    k = 2
    r = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=k)
    c13, s13, g13 = r["q13"]
    c2, s2, g2 = r["q2"]
    ca, sa, ga = O.quantize_nvfp4(I.u16(hidden))
    T = hidden.shape[0]
    Inter = w13.shape[1] // 2
    # amax of h per expert from this loop's own h
    hs = {}
    for t in range(T):
        for j in range(k):
            e = int(r["ids"][t, j])
            g, _ = O.gemm(O.NVFP4, ca[t:t + 1], sa[t:t + 1], ga, c13[e], s13[e], g13[e])
            h = O.silu(g[0, :Inter]) * g[0, Inter:]
            hs[(t, j)] = O.f32_to_bf16_exact(h)
    amax = {}
    for (t, j), h in hs.items():
        e = int(r["ids"][t, j])
        amax[e] = max(amax.get(e, 0.0), float(np.abs(O.bf16_to_f32(h)).max()))
    y = np.zeros((T, hidden.shape[1]))
    for (t, j), h in hs.items():
        e = int(r["ids"][t, j])
        sgh = O.nvfp4_global_scale(amax[e])
        ch, sh = O.quantize_nvfp4_given_scale(h.reshape(1, -1), sgh)
        d, _ = O.gemm(O.NVFP4, ch, sh, sgh, c2[e], s2[e], g2[e])
        y[t] += r["weights"][t, j] * d[0]
    assert np.allclose(r["y"], y, rtol=1e-12, atol=1e-12 * np.abs(y).max())


def test_moe_token_permutation_equivariance(O):
    hidden, logits, w13, w2 = _small_moe(T=8)
    r = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=2)
    perm = np.array([5, 2, 7, 0, 1, 6, 3, 4])
    r2 = O.moe(I.u16(hidden[perm]), logits[perm], I.u16(w13), I.u16(w2), top_k=2, q13=r["q13"], q2=r["q2"])
    assert np.allclose(r2["y"], r["y"][perm], rtol=1e-12, atol=1e-14)


def test_moe_linear_in_down_projection(O):
    """Doubling one expert's W2 doubles its contribution exactly (same codes,
    doubled global scale); zeroing it removes it: y2 + y0 == 2 y."""
    hidden, logits, w13, w2 = _small_moe(T=8)
    base = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=2)
    e = int(base["ids"][0, 0])
    w2x2 = w2.clone()
    w2x2[e] = w2[e] * 2
    w2x0 = w2.clone()
    w2x0[e] = 0
    y2 = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2x2), top_k=2, q13=base["q13"])["y"]
    y0 = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2x0), top_k=2, q13=base["q13"])["y"]
    assert np.allclose(y2 + y0, 2 * base["y"], rtol=1e-12, atol=1e-14)
    assert not np.allclose(y0, base["y"])


def test_moe_single_expert_is_two_linears(O):
    hidden, logits, w13, w2 = _small_moe(E=1, k=1)
    r = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=1)
    assert np.allclose(r["weights"], 1.0)
    g, _, _, _ = O.linear(O.NVFP4, I.u16(hidden), I.u16(w13[0]))
    Inter = w13.shape[1] // 2
    h = O.f32_to_bf16_exact(O.silu(g[:, :Inter]) * g[:, Inter:])
    y, _, _, _ = O.linear(O.NVFP4, h, I.u16(w2[0]))
    assert np.allclose(r["y"], y, rtol=1e-12, atol=1e-14)


def test_moe_static_scales_path(O):
    hidden, logits, w13, w2 = _small_moe()
    E = 4
    st13 = np.full(E, 3.0 / 2688, dtype=np.float32)
    st2 = np.full(E, 0.05 / 2688, dtype=np.float32)
    r = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=2, mode=O.STATIC, static13=st13, static2=st2)
    assert np.all(r["sgH"][r["counts"] > 0] == st2[0])
    assert np.isfinite(r["y"]).all() and np.abs(r["y"]).max() > 0


# ---------------------------------------------- MoE with per-expert static scales
#
# "GLM-5.3-Flash on vLLM, on GB10", the account of the uninitialised MoE
# activation scale: a checkpoint's per-expert input_scale sets each expert's
# activation global scale, and alpha = weight_scale_2 x input_scale.  The pins
# below use a DIFFERENT scale per expert (and different scales for the two
# GEMMs), so a swapped pair of arrays or a wrong expert index fails them.

def _distinct_static_scales(E):
    rng = np.random.default_rng(41)
    st13 = (rng.permutation(np.linspace(1.5, 6.0, E)) / 2688).astype(np.float32)
    st2 = (rng.permutation(np.linspace(0.2, 0.9, E)) / 2688).astype(np.float32)
    assert len(set(st13.tolist())) == E and len(set(st2.tolist())) == E
    assert not set(st13.tolist()) & set(st2.tolist())
    return st13, st2


def test_moe_static_per_token_loop(O):
    """Static mode against a loop over (token, slot): the token's row is
    quantised under its expert's static13[e], GEMM1 takes alpha1 = static13[e]
    x s_gW13[e], h is requantised under static2[e] and GEMM2 takes alpha2 =
    static2[e] x s_gW2[e]; the combine sums the k terms by routing weight."""
    hidden, logits, w13, w2 = _small_moe(T=7, E=4, k=2)
    k, E = 2, 4
    st13, st2 = _distinct_static_scales(E)
    r = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=k, mode=O.STATIC, static13=st13, static2=st2)
    c13, s13, g13 = r["q13"]
    c2, s2, g2 = r["q2"]
    T = hidden.shape[0]
    Inter = w13.shape[1] // 2
    pos = np.empty(T * k, dtype=np.int64)
    pos[r["order"]] = np.arange(T * k)
    y = np.zeros((T, hidden.shape[1]))
    hu = I.u16(hidden)
    for t in range(T):
        for j in range(k):
            e = int(r["ids"][t, j])
            ca, sa = O.quantize_nvfp4_given_scale(hu[t:t + 1], st13[e])
            assert np.array_equal(r["a_codes"][pos[t * k + j]], ca[0])
            assert np.array_equal(r["a_scales"][pos[t * k + j]], sa[0])
            g, _ = O.gemm(O.NVFP4, ca, sa, st13[e], c13[e], s13[e], g13[e])
            h = O.f32_to_bf16_exact(O.silu(g[0, :Inter]) * g[0, Inter:]).reshape(1, -1)
            ch, sh = O.quantize_nvfp4_given_scale(h, st2[e])
            assert np.array_equal(r["h_codes"][pos[t * k + j]], ch[0])
            d, _ = O.gemm(O.NVFP4, ch, sh, st2[e], c2[e], s2[e], g2[e])
            y[t] += r["weights"][t, j] * d[0]
    assert np.allclose(r["y"], y, rtol=1e-12, atol=1e-12 * np.abs(y).max())
    used = r["counts"] > 0
    assert np.array_equal(r["sgH"][used], st2[used])


def test_moe_static_scale_locality(O):
    """Changing one expert's static13 changes only the dispatched rows of that
    expert and the outputs of the tokens routed to it; the same for static2
    and the requantised h.  Exchanging the two arrays changes the result."""
    hidden, logits, w13, w2 = _small_moe(T=9, E=4, k=2)
    k, E = 2, 4
    st13, st2 = _distinct_static_scales(E)
    kw = dict(top_k=k, mode=O.STATIC)
    base = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), static13=st13, static2=st2, **kw)
    q = dict(q13=base["q13"], q2=base["q2"])
    offs = base["offsets"]
    tok = base["order"] // k
    for e0 in range(E):
        lo, hi = offs[e0], offs[e0 + 1]
        if hi == lo:
            continue
        routed = np.zeros(hidden.shape[0], dtype=bool)
        routed[np.unique(tok[lo:hi])] = True
        rows_other = np.r_[0:lo, hi:offs[-1]]
        s = st13.copy()
        s[e0] *= 1.37
        r = O.moe(I.u16(hidden), logits, static13=s, static2=st2, **q, **kw)
        assert np.array_equal(r["a_codes"][rows_other], base["a_codes"][rows_other])
        assert not np.array_equal(r["a_codes"][lo:hi], base["a_codes"][lo:hi])
        assert np.array_equal(r["y"][~routed], base["y"][~routed])
        assert not np.allclose(r["y"][routed], base["y"][routed])
        s = st2.copy()
        s[e0] *= 1.37
        r = O.moe(I.u16(hidden), logits, static13=st13, static2=s, **q, **kw)
        assert np.array_equal(r["a_codes"], base["a_codes"])
        assert np.array_equal(r["h_codes"][rows_other], base["h_codes"][rows_other])
        assert not np.array_equal(r["h_codes"][lo:hi], base["h_codes"][lo:hi])
        assert np.array_equal(r["y"][~routed], base["y"][~routed])
        assert not np.allclose(r["y"][routed], base["y"][routed])
    swapped = O.moe(I.u16(hidden), logits, static13=st2, static2=st13, **q, **kw)
    assert not np.allclose(swapped["y"], base["y"])


def test_moe_static_exact_dispatch_round_trip(O):
    """Hidden blocks on the E2M1 grid times a power of two (block maximum
    6 x 2^j) and power-of-two static13 scales that differ per expert: every
    dispatched row then dequantises to the hidden row exactly (the block
    scale is 2^j / static13[e], an E4M3 power of two), so GEMM1's G equals the
    fp64 product of the hidden rows with the dequantised W13 of the row's
    expert, whatever static13[e] is: the per-expert scale cancels between the
    quantiser and alpha1."""
    T, E, k, H, Inter = 6, 4, 2, 64, 32
    _, logits, w13, w2 = _small_moe(T=T, E=E, H=H, Inter=Inter, k=k)
    rng = np.random.default_rng(5)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    x = rng.choice(grid, size=(T, H)) * rng.choice([-1, 1], size=(T, H))
    x[:, ::16] = 6.0  # each 16-element block holds its maximum 6
    x *= np.repeat(2.0 ** rng.integers(-3, 4, size=(T, H // 16)), 16, axis=1)
    hidden = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(hidden.double().numpy(), x)
    st13 = np.array([2.0 ** -3, 2.0 ** -5, 2.0 ** -1, 2.0 ** -4], dtype=np.float32)
    st2 = np.full(E, 0.5 / 2688, dtype=np.float32)
    r = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=k, mode=O.STATIC, static13=st13, static2=st2)
    c13, s13, g13 = r["q13"]
    tok = r["order"] // k
    for e in range(E):
        lo, hi = r["offsets"][e], r["offsets"][e + 1]
        if hi == lo:
            continue
        deq = O.dequantize(O.NVFP4, r["a_codes"][lo:hi], r["a_scales"][lo:hi], st13[e])
        assert np.array_equal(deq, x[tok[lo:hi]])
        w = O.dequantize(O.NVFP4, c13[e], s13[e], g13[e])
        assert np.allclose(r["G"][lo:hi], x[tok[lo:hi]] @ w.T, rtol=1e-12, atol=1e-12)


def test_moe_static_scale_far_below_amax_saturates(O):
    """A static scale far below amax / 2688 saturates: every block scale of the
    expert's dispatched rows is E4M3 448 (byte 0x7E) and every nonzero element
    is E2M1 +-6 (codes 0x7 / 0xF); the other experts' rows are unaffected."""
    hidden, logits, w13, w2 = _small_moe(T=8, E=4, k=2)
    k, E = 2, 4
    st13, st2 = _distinct_static_scales(E)
    base = O.moe(I.u16(hidden), logits, I.u16(w13), I.u16(w2), top_k=k, mode=O.STATIC, static13=st13,
                 static2=st2)
    e0 = int(np.argmax(base["counts"]))
    s = st13.copy()
    s[e0] = 1e-12
    r = O.moe(I.u16(hidden), logits, top_k=k, mode=O.STATIC, static13=s, static2=st2, q13=base["q13"],
              q2=base["q2"])
    lo, hi = r["offsets"][e0], r["offsets"][e0 + 1]
    assert hi > lo
    assert np.all(r["a_scales"][lo:hi] == 0x7E)
    codes = r["a_codes"][lo:hi]
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(hi - lo, -1)
    xs = I.u16(hidden)[r["order"][lo:hi] // k]
    nonzero = (xs & 0x7FFF) != 0
    assert np.all((nib[nonzero] & 7) == 7)
    assert np.array_equal((nib >> 3).astype(bool)[nonzero], (xs >> 15).astype(bool)[nonzero])
    rest = np.r_[0:lo, hi:r["offsets"][-1]]
    assert np.array_equal(r["a_codes"][rest], base["a_codes"][rest])
