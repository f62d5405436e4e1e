"""GPU MXFP8 / MXFP6 against the CPU oracle (oracle.mx_wide).

Quantisers (E4M3, E5M2, E2M3, E3M2 elements): codes and the whole scale
buffer (padding included) bit for bit.  MXFP8 GEMM (E4M3 / E5M2 operands,
tcgen05 kind::mxf8f6f4): every output element, or sampled rows and columns at
the full prefill size, within the tolerance of tests/util.py (no global
scale: alpha = 1).  MXFP6: the exact widening of every 6-bit code to E4M3,
and MXFP6 (or mixed) linears through the E4M3 GEMM against the oracle's
products of the 6-bit values."""
import numpy as np
import pytest
import torch

from mxfp4_block_scaled_gb300 import inputs as I
from oracle import mx_wide as X
from util import bf16_to_np, check_close

pytestmark = pytest.mark.gpu

ELEMS = [0, 1, 2, 3]  # FP4_MX_E4M3, FP4_MX_E5M2, FP4_MX_E2M3, FP4_MX_E3M2
NAME = {0: "e4m3", 1: "e5m2", 2: "e2m3", 3: "e3m2"}


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__ as ge
    ge.build()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


def _dev(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()


def check(F, O, u16, elem=0):
    rows, k = u16.shape
    x = _dev(u16)
    if elem == 0:
        codes, scales = F.quantize_mxfp8(x)
    else:
        q = F.quantize_mx(x, elem)
        codes, scales = q.codes, q.scales
    torch.cuda.synchronize()
    F.device_status()
    want_c, want_s = X.quantize(NAME[elem], u16)
    assert np.array_equal(codes.cpu().numpy(), want_c.astype(np.uint8))
    assert np.array_equal(scales.cpu().numpy(), O.scales_to_mma(want_s, rows, k, O.MXFP4))


# ragged rows (scale-layout padding to 128), k not a multiple of 256, one block, several tiles
@pytest.mark.parametrize("rows,k", [(1, 32), (3, 96), (130, 800), (257, 4096), (64, 7168)])
@pytest.mark.parametrize("elem", ELEMS)
def test_mx_quant_shapes(F, O, rows, k, elem):
    check(F, O, I.u16(I.activations_with_outliers(rows, k, rows + k)), elem)


@pytest.mark.parametrize("elem", ELEMS)
def test_mx_quant_adversarial(F, O, elem):
    """Exact midpoints of the element grid (ties to even), their bf16
    neighbours, signed zeros, bf16 subnormals, values near the bf16 maximum,
    all-zero blocks and blocks whose amax is an exact power of two."""
    rng = np.random.default_rng(9 + elem)
    rows, k = 8, 256
    u = I.u16(I.randn_bf16((rows, k), 17)).copy()
    _, g = X.grid(NAME[elem])
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)
    top = np.float32(g[-1])
    # row 0: block max = the largest element (scale 2^0 when it is a power of
    # two's multiple), then midpoints and their bf16 neighbours
    row0 = np.concatenate([[top], rng.choice(mids, 31)]).astype(np.float32)
    row0 = row0 * np.where(rng.random(32) < 0.5, -1, 1).astype(np.float32)
    u[0, :32] = (row0.view(np.uint32) >> 16).astype(np.uint16)
    u[0, 32:64] = u[0, :32] + 1
    u[0, 64:96] = u[0, :32] - 1
    u[1, :32] = 0x8000                                # negative zeros
    u[1, 32:64] = 0                                   # zeros
    u[1, 64:96] = rng.integers(1, 0x80, 32)           # positive bf16 subnormals
    u[1, 96:128] = rng.integers(0x8001, 0x8080, 32)   # negative bf16 subnormals
    u[2, :32] = rng.integers(0x7F00, 0x7F80, 32)      # near the bf16 maximum
    u[2, 32:64] = np.uint16(0x4000)                   # all 2.0
    u[2, 64:96] = 0x8000
    u[2, 64] = np.uint16(0x3F80)                      # one 1.0 among negative zeros
    # row 3: a block of values just below the saturation threshold times 2^e
    sat = (np.float32(top) * np.float32(1.0 + 2.0 ** -5)).astype(np.float32)
    u[3, :32] = (np.full(32, sat, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    u[3, 5] = (np.array([top], dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)[0]
    check(F, O, u, elem)


def test_mxfp8_full_size(F, O):
    """The prefill activation shape, 2048 rows of K = 4096 (every code)."""
    check(F, O, I.u16(I.randn_bf16((2048, 4096), 2)))


@pytest.mark.parametrize("elem", [1, 2, 3])
def test_mx_quant_full_size(F, O, elem):
    check(F, O, I.u16(I.randn_bf16((1024, 4096), 2 + elem)), elem)


# ------------------------------------------------------------------ GEMM

def mx_linear(F, a, w, ea, ew):
    """GPU: weights quantised by fp4_quantize_mx, activations per call by
    fp4_gemm_mx; oracle: both quantised by mx_wide, then its fp64 GEMM."""
    wq = F.quantize_mx(w.cuda(), ew)
    got = bf16_to_np(F.gemm_mx(a.cuda(), wq, ea))
    torch.cuda.synchronize()
    F.device_status()
    ca, sa = X.quantize(NAME[ea], I.u16(a))
    cw, sw = X.quantize(NAME[ew], I.u16(w))
    ref, mag = X.gemm(NAME[ea], ca, sa, NAME[ew], cw, sw)
    return got, ref, mag


# (m, n, k): one tile, ragged M / N / K tails, k not a multiple of 128, several waves
MX_SHAPES = [(1, 256, 512), (33, 264, 800), (128, 256, 256), (130, 520, 1056), (300, 1280, 2048),
             (512, 2048, 544)]


@pytest.mark.parametrize("m,n,k", MX_SHAPES)
@pytest.mark.parametrize("ea,ew", [(0, 0), (1, 1), (0, 1), (1, 0)])
def test_mx_gemm_shapes(F, O, m, n, k, ea, ew):
    a = I.randn_bf16((m, k), m + n + ea)
    w = I.weights_bf16(n, k, k + 3 + ew)
    got, ref, mag = mx_linear(F, a, w, ea, ew)
    check_close(got, ref, mag)


def test_mx_gemm_prequant_matches_per_call(F, O):
    """fp4_gemm_mx_prequant on operands quantised by fp4_quantize_mx gives the
    same bits as fp4_gemm_mx (which quantises the activations itself)."""
    a = I.randn_bf16((200, 1024), 5).cuda()
    w = I.weights_bf16(384, 1024, 6).cuda()
    wq = F.quantize_mx(w, 1)
    o1 = F.gemm_mx(a, wq, 0)
    o2 = F.gemm_mx_prequant(F.quantize_mx(a, 0), wq)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("elem", [2, 3])
def test_mx_widen_is_exact(F, O, elem):
    """Every 6-bit code (both signs) widens to the E4M3 code of the same
    value, in place and out of place."""
    codes = np.tile(np.arange(64, dtype=np.uint8), 32).reshape(4, 512)
    q = F.MXTensor(elem, 4, 512, torch.from_numpy(codes).cuda(), torch.zeros(512, dtype=torch.uint8, device="cuda"))
    wide = F.mx_widen(q).codes.cpu().numpy()
    want = X.decode(NAME[elem], codes.astype(np.int64))
    got = X.decode("e4m3", wide.astype(np.int64))
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))  # -0 stays -0
    F.lib().fp4_mx_widen(elem, q.codes.data_ptr(), 4, 512, q.codes.data_ptr(), None)  # in place
    torch.cuda.synchronize()
    assert np.array_equal(q.codes.cpu().numpy(), wide)


def mx6_linear(F, a, w, ea, ew):
    """MXFP6 (or mixed) linear: W quantised to ew and, if MXFP6, widened;
    activations quantised to ea per call by fp4_gemm_mx."""
    wq = F.quantize_mx(w.cuda(), ew)
    if ew >= 2:
        wq = F.mx_widen(wq)
    got = bf16_to_np(F.gemm_mx(a.cuda(), wq, ea))
    torch.cuda.synchronize()
    F.device_status()
    ca, sa = X.quantize(NAME[ea], I.u16(a))
    cw, sw = X.quantize(NAME[ew], I.u16(w))
    ref, mag = X.gemm(NAME[ea], ca, sa, NAME[ew], cw, sw)
    return got, ref, mag


@pytest.mark.parametrize("m,n,k", [(1, 256, 512), (33, 264, 800), (130, 520, 1056), (300, 1280, 2048)])
@pytest.mark.parametrize("ea,ew", [(2, 2), (3, 3), (2, 3), (0, 2), (3, 1)])
def test_mxfp6_gemm_shapes(F, O, m, n, k, ea, ew):
    """MXFP6 operands through the E4M3 GEMM after the exact widening: the
    products are those of the MXFP6 values (the oracle computes them from the
    6-bit codes)."""
    a = I.randn_bf16((m, k), m + n + 7 * ea)
    w = I.weights_bf16(n, k, k + 5 + ew)
    got, ref, mag = mx6_linear(F, a, w, ea, ew)
    check_close(got, ref, mag)


def test_mx_gemm_refuses_unwidened_fp6(F, O):
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    wq = F.quantize_mx(torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda"), 2)
    with pytest.raises(F.FP4Error) as e:
        F.gemm_mx(x, wq, 0)
    assert e.value.name == "FP4_ERR_INVALID_ARG"
    with pytest.raises(F.FP4Error):
        F.gemm_mx_prequant(F.quantize_mx(x, 2), F.mx_widen(wq))


def test_mxfp8_prefill_full_size_sampled(F, O):
    """MXFP8 (E4M3 x E4M3) at the prefill shape M=8192, K=4096, N=14336: all
    columns of sampled rows and all rows of sampled columns."""
    m, k, n = 8192, 4096, 14336
    a = I.randn_bf16((m, k), 2)
    w = I.weights_bf16(n, k, 102)
    wq = F.quantize_mx(w.cuda(), 0)
    got = bf16_to_np(F.gemm_mx(a.cuda(), wq, 0))
    torch.cuda.synchronize()
    F.device_status()
    ca, sa = X.quantize("e4m3", I.u16(a))
    cw, sw = X.quantize("e4m3", I.u16(w))
    rng = np.random.default_rng(n)
    rows = np.unique(np.concatenate([rng.choice(m, 24, replace=False), [0, 127, 128, m - 1]]))
    cols = np.unique(np.concatenate([rng.choice(n, 12, replace=False), [0, 255, 256, n - 1]]))
    ref, mag = X.gemm("e4m3", ca[rows], sa[rows], "e4m3", cw, sw)
    check_close(got[rows], ref, mag, what="sampled rows")
    ref, mag = X.gemm("e4m3", ca, sa, "e4m3", cw[cols], sw[cols])
    check_close(got[:, cols], ref, mag, what="sampled columns")
