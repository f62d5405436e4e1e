"""GPU block-scaled GEMM vs the CPU oracle's dequantise-then-fp64 GEMM.

The oracle quantises the same bf16 inputs itself (its codes are checked bit
for bit against the GPU quantiser elsewhere) and computes the reference and
the magnitude sum that sizes the fp32 accumulation floor; see tests/util.py
for the tolerance."""
import numpy as np
import pytest
import torch

from mxfp4_block_scaled_gb300 import inputs as I
from util import bf16_to_np, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__ as ge
    ge.build()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


def run_gemm(F, a, w, fmt, mode=0, st=0.0):
    wq = F.prepack_weight(w.cuda(), fmt)
    out = F.gemm(a.cuda(), wq, mode, st)
    torch.cuda.synchronize()
    F.device_status()
    return bf16_to_np(out)


def check_linear(F, O, a, w, fmt, mode=0, st=0.0):
    got = run_gemm(F, a, w, fmt, mode, st)
    ref, mag, _, _ = O.linear(fmt, I.u16(a), I.u16(w), mode, st)
    check_close(got, ref, mag)


def test_single_linear_workload(F, O):
    """A [16, 512] ~ N(0,1) seed 0, W [256, 512] ~ N(0, 0.02), NVFP4 dynamic."""
    check_linear(F, O, I.randn_bf16((16, 512), 0), I.weights_bf16(256, 512, 100), 0)


# (m, n, k): several tiles, ragged M / N / K tails, both the prefill (m > 64)
# and the weight-streaming decode (m <= 64, split-K) paths.
SHAPES = [(1, 256, 512), (3, 1024, 768), (8, 520, 1024), (32, 1024, 4096), (33, 264, 512), (64, 384, 256),
          (65, 264, 800), (128, 256, 256), (130, 520, 1056), (300, 1280, 2048), (512, 2048, 512)]


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("fmt", [0, 1])
def test_shapes(F, O, m, n, k, fmt):
    check_linear(F, O, I.randn_bf16((m, k), m + n), I.weights_bf16(n, k, k + 3), fmt)


# the CTA-pair kernel (forced by the tile policy): more pair tiles than SMs,
# a ragged M whose last pair tile has an empty odd half, a ragged N, and
# problems of one or two pair tiles
@pytest.mark.parametrize("m,n,k", [(2660, 4096, 512), (2395, 4104, 768), (256, 256, 256), (300, 520, 1056)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_pair_kernel_shapes(F, O, m, n, k, fmt):
    F.set_gemm_tile_policy(F.TILE_CTA_PAIR)
    try:
        check_linear(F, O, I.randn_bf16((m, k), m), I.weights_bf16(n, k, n), fmt)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)


# the fused decode kernel (activation quantisation inside the GEMM launch),
# forced on small and ragged shapes: n not a multiple of 128, k not of 256;
# the ring depth follows m and k (k = 8192 at m = 8: 7 stages, 32 K blocks)
@pytest.mark.parametrize("m,n,k", [(1, 256, 512), (5, 520, 800), (8, 1000, 1056), (3, 128, 4096), (8, 384, 8192),
                                   (1, 256, 8192)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_fused_decode_shapes(F, O, m, n, k, fmt):
    F.set_gemm_tile_policy(F.TILE_FUSED_DECODE)
    try:
        check_linear(F, O, I.activations_with_outliers(m, k, m + k), I.weights_bf16(n, k, n + 7), fmt)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)


def test_fused_decode_static_scale(F, O):
    F.set_gemm_tile_policy(F.TILE_FUSED_DECODE)
    try:
        a = I.randn_bf16((4, 1024), 21)
        w = I.weights_bf16(640, 1024, 22)
        check_linear(F, O, a, w, 0, mode=1, st=3.5 / 2688)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)


def test_static_scale(F, O):
    a = I.randn_bf16((96, 512), 9)
    w = I.weights_bf16(256, 512, 10)
    check_linear(F, O, a, w, 0, mode=1, st=3.5 / 2688)   # clips the largest activations
    check_linear(F, O, a[:8], w, 0, mode=1, st=0.02)


def test_prequant_with_oracle_operands(F, O):
    """The GEMM alone, on operands quantised by the oracle and uploaded."""
    for fmt, (m, n, k) in [(0, (200, 512, 1024)), (1, (200, 512, 1024)), (0, (5, 640, 2048))]:
        a = I.randn_bf16((m, k), 1)
        w = I.weights_bf16(n, k, 2)
        ca, sa, ga = O.quantize(fmt, I.u16(a))
        cw, sw, gw = O.quantize(fmt, I.u16(w))
        ref, mag = O.gemm(fmt, ca, sa, ga, cw, sw, gw)

        def up(c, s, g, rows):
            q = F.empty_qtensor(fmt, rows, k, "cuda")
            q.codes.copy_(torch.from_numpy(c))
            q.scales.copy_(torch.from_numpy(O.scales_to_mma(s, rows, k, fmt)))
            q.gscale.fill_(float(g))
            return q

        out = F.gemm_prequant(up(ca, sa, ga, m), up(cw, sw, gw, n))
        torch.cuda.synchronize()
        check_close(bf16_to_np(out), ref, mag)


def test_zero_m_is_noop(F):
    w = I.weights_bf16(256, 512, 1).cuda()
    wq = F.prepack_weight(w)
    out = F.gemm(torch.empty((0, 512), dtype=torch.bfloat16, device="cuda"), wq)
    torch.cuda.synchronize()
    assert out.shape == (0, 256)


def test_zero_activations_give_zero(F):
    w = I.weights_bf16(256, 512, 1).cuda()
    out = F.gemm(torch.zeros((40, 512), dtype=torch.bfloat16, device="cuda"), F.prepack_weight(w))
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()


# ------------------------------------------------------------ full sizes

@pytest.fixture(scope="module")
def decode_weights(O):
    w = I.weights_bf16(14336, 4096, 101)
    return w, O.quantize_nvfp4(I.u16(w))


@pytest.mark.parametrize("m", [1, 8, 32])
def test_decode_full_size(F, O, decode_weights, m):
    """Decode-shaped NVFP4 GEMM: K=4096, N=14336, activations with 0.1%
    outliers x50; every output element checked."""
    w, qw = decode_weights
    a = I.activations_with_outliers(m, 4096, 1)
    got = run_gemm(F, a, w, 0)
    qa = O.quantize_nvfp4(I.u16(a))
    ref, mag = O.gemm(0, qa[0], qa[1], qa[2], *qw)
    check_close(got, ref, mag)


@pytest.mark.parametrize("n", [4096, 14336])
def test_prefill_full_size_sampled(F, O, n):
    """Prefill-shaped NVFP4 GEMM M=8192, K=4096: all columns of 48 sampled
    rows and all rows of 24 sampled columns (rows/cols span every tile)."""
    m, k = 8192, 4096
    a = I.randn_bf16((m, k), 2)
    w = I.weights_bf16(n, k, 102)
    got = run_gemm(F, a, w, 0)
    qa = O.quantize_nvfp4(I.u16(a))
    qw = O.quantize_nvfp4(I.u16(w))
    rng = np.random.default_rng(n)
    rows = np.unique(np.concatenate([rng.choice(m, 40, replace=False), [0, 127, 128, m - 1]]))
    cols = np.unique(np.concatenate([rng.choice(n, 20, replace=False), [0, 255, 256, n - 1]]))
    ref, mag = O.gemm_rows(0, qa[0], qa[1], qa[2], qw[0], qw[1], qw[2], rows, np.arange(n))
    check_close(got[rows], ref, mag, what="sampled rows")
    ref, mag = O.gemm_rows(0, qa[0], qa[1], qa[2], qw[0], qw[1], qw[2], np.arange(m), cols)
    check_close(got[:, cols], ref, mag, what="sampled columns")


def test_prefill_full_size_weight_pairs(F, O):
    """The prefill shape on the weight-tile-sharing CTA pairs: sampled rows and
    columns as above, and the same bits as the one-CTA kernel (the MMAs and
    the epilogue are the same; only the copies that feed them differ)."""
    m, k, n = 8192, 4096, 14336
    a = I.randn_bf16((m, k), 2)
    w = I.weights_bf16(n, k, 102)
    base = run_gemm(F, a, w, 0)
    F.set_gemm_tile_policy(F.TILE_WEIGHT_PAIRS)
    try:
        assert F.plan_gemm(m, n, k, torch.cuda.get_device_properties(0).multi_processor_count)["weight_pairs"]
        got = run_gemm(F, a, w, 0)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)
    assert np.array_equal(got, base)
    qa = O.quantize_nvfp4(I.u16(a))
    qw = O.quantize_nvfp4(I.u16(w))
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(m, 24, replace=False), [0, 127, 128, 255, 256, m - 1]]))
    cols = np.unique(np.concatenate([rng.choice(n, 12, replace=False), [0, 127, 128, 255, 256, n - 1]]))
    ref, mag = O.gemm_rows(0, qa[0], qa[1], qa[2], qw[0], qw[1], qw[2], rows, np.arange(n))
    check_close(got[rows], ref, mag, what="sampled rows")
    ref, mag = O.gemm_rows(0, qa[0], qa[1], qa[2], qw[0], qw[1], qw[2], np.arange(m), cols)
    check_close(got[:, cols], ref, mag, what="sampled columns")


# the one-CTA kernel in clusters of two whose activation tiles share each
# 256-row weight tile (TMA multicast of its halves), forced: whole pairs of
# activation tiles, ragged N and K, one and several pair units per cluster
@pytest.mark.parametrize("m,n,k", [(1024, 5120, 512), (1280, 4904, 1056), (2048, 10240, 256)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_weight_pair_kernel_shapes(F, O, m, n, k, fmt):
    F.set_gemm_tile_policy(F.TILE_WEIGHT_PAIRS)
    try:
        assert F.plan_gemm(m, n, k, torch.cuda.get_device_properties(0).multi_processor_count)["weight_pairs"]
        check_linear(F, O, I.randn_bf16((m, k), m + 5), I.weights_bf16(n, k, n + 11), fmt)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)


def test_mxfp4_full_size(F, O):
    """MXFP4 W4A4 M=2048, K=7168, N=2048: every output element."""
    a = I.randn_bf16((2048, 7168), 4)
    w = I.weights_bf16(2048, 7168, 104)
    check_linear(F, O, a, w, 1)


# ------------------------------------------------------ weight-only (W4A16)

def check_w4a16(F, O, x, w, fmt, qw=None):
    wq = F.prepack_weight(w.cuda(), fmt)
    got = bf16_to_np(F.gemm_w4a16(x.cuda(), wq))
    torch.cuda.synchronize()
    F.device_status()
    cw, sw, gw = qw if qw is not None else O.quantize(fmt, I.u16(w))
    ref, mag = O.linear_w4a16(fmt, I.u16(x), cw, sw, gw)
    check_close(got, ref, mag)


# ragged rows of codes (k = 800: a partial 512-byte warp load), the one-lane
# row (k = 32), rows per CTA not dividing n, and the wide-row kernel
# (k > 4096: up to eight warp loads per row, k = 4128 needs five)
@pytest.mark.parametrize("m,n,k", [(1, 256, 512), (2, 520, 800), (3, 1000, 1056), (4, 264, 4096), (1, 8, 32),
                                   (2, 1032, 4128), (4, 128, 8192)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_w4a16_shapes(F, O, m, n, k, fmt):
    check_w4a16(F, O, I.activations_with_outliers(m, k, m + 5 * k), I.weights_bf16(n, k, n + 11), fmt)


@pytest.mark.parametrize("m,n,k", [(1, 256, 512), (2, 520, 800), (3, 1000, 1056), (4, 264, 4096), (1, 8, 32),
                                   (2, 1032, 4128), (4, 128, 8192)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_w4a16_tensor_core_shapes(F, O, m, n, k, fmt):
    """The same shapes forced onto the tensor-core kernel (weights dequantised
    to bf16 in shared memory, kind::f16 MMAs): ragged n and k, one K block."""
    F.set_gemm_tile_policy(F.TILE_W4A16_TC)
    try:
        check_w4a16(F, O, I.activations_with_outliers(m, k, m + 5 * k), I.weights_bf16(n, k, n + 11), fmt)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)


def test_w4a16_tensor_core_mxfp4_full_size(F, O):
    """MXFP4 W [4096, 7168], m = 3, on the tensor-core kernel."""
    F.set_gemm_tile_policy(F.TILE_W4A16_TC)
    try:
        check_w4a16(F, O, I.activations_with_outliers(3, 7168, 6), I.weights_bf16(4096, 7168, 105), 1)
    finally:
        F.set_gemm_tile_policy(F.TILE_AUTO)


def test_w4a16_empty_and_zero(F):
    w = I.weights_bf16(256, 512, 1).cuda()
    wq = F.prepack_weight(w)
    assert F.gemm_w4a16(torch.empty((0, 512), dtype=torch.bfloat16, device="cuda"), wq).shape == (0, 256)
    out = F.gemm_w4a16(torch.zeros((3, 512), dtype=torch.bfloat16, device="cuda"), wq)
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()


def test_w4a16_rejects_five_rows(F):
    wq = F.prepack_weight(I.weights_bf16(256, 512, 1).cuda())
    with pytest.raises(F.FP4Error):
        F.gemm_w4a16(torch.zeros((5, 512), dtype=torch.bfloat16, device="cuda"), wq)


@pytest.mark.parametrize("m", [1, 4])
def test_w4a16_full_size(F, O, decode_weights, m):
    """Weight-only decode, NVFP4 W [14336, 4096], activations with 0.1%
    outliers x50: every output element."""
    w, qw = decode_weights
    check_w4a16(F, O, I.activations_with_outliers(m, 4096, 3), w, 0, qw)


def test_w4a16_mxfp4_full_size(F, O):
    """Weight-only decode, MXFP4 W [4096, 7168], m = 2: every output element."""
    check_w4a16(F, O, I.activations_with_outliers(2, 7168, 5), I.weights_bf16(4096, 7168, 105), 1)
