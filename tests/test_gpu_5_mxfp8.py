"""GPU MXFP8 (E4M3) quantiser vs the CPU oracle: codes and the whole scale
buffer (padding included) bit for bit."""
import numpy as np
import pytest
import torch

from mxfp4_block_scaled_gb300 import inputs as I
from oracle import mx_wide as X

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__ as ge
    ge.build()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


def check(F, O, u16):
    rows, k = u16.shape
    x = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()
    codes, scales = F.quantize_mxfp8(x)
    torch.cuda.synchronize()
    F.device_status()
    want_c, want_s = X.quantize("e4m3", u16)
    assert np.array_equal(codes.cpu().numpy(), want_c.astype(np.uint8))
    assert np.array_equal(scales.cpu().numpy(), O.scales_to_mma(want_s, rows, k, O.MXFP4))


# ragged rows (scale-layout padding to 128), k not a multiple of 256, one block, several tiles
@pytest.mark.parametrize("rows,k", [(1, 32), (3, 96), (130, 800), (257, 4096), (64, 7168)])
def test_mxfp8_shapes(F, O, rows, k):
    check(F, O, I.u16(I.activations_with_outliers(rows, k, rows + k)))


def test_mxfp8_adversarial(F, O):
    """Exact midpoints of the E4M3 grid (ties to even), their bf16
    neighbours, signed zeros, bf16 subnormals, values near the bf16 maximum,
    all-zero blocks and blocks whose amax is an exact power of two."""
    rng = np.random.default_rng(9)
    rows, k = 8, 256
    u = I.u16(I.randn_bf16((rows, k), 17)).copy()
    _, g = X.grid("e4m3")
    mids = ((g[1:] + g[:-1]) / 2).astype(np.float32)
    # row 0: block max 448 (scale 2^0), then midpoints and their bf16 neighbours
    row0 = np.concatenate([[448.0], rng.choice(mids, 31)]).astype(np.float32)
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
    check(F, O, u)


def test_mxfp8_full_size(F, O):
    """The prefill activation shape, 2048 rows of K = 4096 (every code)."""
    check(F, O, I.u16(I.randn_bf16((2048, 4096), 2)))
