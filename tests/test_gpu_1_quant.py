"""GPU quantiser vs the CPU oracle: codes, scales (whole MMA-layout buffer,
padding included) and the global scale must match bit for bit."""
import numpy as np
import pytest
import torch

from mxfp4_block_scaled_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__ as ge
    ge.build()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


def gpu_quant(F, x, fmt, mode=0, st=0.0):
    q = F.quantize(x.cuda(), fmt, mode, st)
    torch.cuda.synchronize()
    F.device_status()
    return q.codes.cpu().numpy(), q.scales.cpu().numpy(), float(q.gscale.cpu()[0])


def check_quant(F, O, x, fmt, mode=0, st=0.0):
    rows, k = x.shape
    c_g, s_g, g_g = gpu_quant(F, x, fmt, mode, st)
    c_o, s_o, g_o = O.quantize(fmt, I.u16(x), mode, st)
    s_o_mma = O.scales_to_mma(s_o, rows, k, fmt)
    assert np.float32(g_g).tobytes() == np.float32(g_o).tobytes(), (g_g, g_o)
    bad = np.nonzero(c_g != c_o)
    assert bad[0].size == 0, "codes differ at %d places, first %s: gpu %s oracle %s" % (
        bad[0].size, (bad[0][0], bad[1][0]), hex(c_g[bad][0]), hex(c_o[bad][0]))
    bads = np.nonzero(s_g != s_o_mma)[0]
    assert bads.size == 0, "scales differ at %d bytes, first %d: gpu %s oracle %s" % (
        bads.size, bads[0], hex(s_g[bads[0]]), hex(s_o_mma[bads[0]]))


SHAPES = [(1, 32), (3, 64), (16, 512), (130, 800), (257, 4096), (128, 256)]


@pytest.mark.parametrize("rows,k", SHAPES)
@pytest.mark.parametrize("fmt", [0, 1])
def test_random_normal(F, O, rows, k, fmt):
    check_quant(F, O, I.randn_bf16((rows, k), rows * 7 + k), fmt)


@pytest.mark.parametrize("st", [1.0, 0.01, 3.0e-3, 1e-30, 5.5 / 2688])
def test_nvfp4_static(F, O, st):
    check_quant(F, O, I.randn_bf16((64, 512), 5), 0, mode=1, st=st)


def test_decode_outliers(F, O):
    for m in (1, 8, 32):
        check_quant(F, O, I.activations_with_outliers(m, 4096, 1), 0)


def _adversarial(k=512):
    """Rows that hit every rounding tie, zeros, signed zeros, subnormals,
    saturation and tiny / huge blocks."""
    rows = []
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    # ties with a block scale of exactly 2 (static s_g = 1): block amax 12
    r = np.zeros(k, np.float32)
    for b in range(k // 16):
        r[b * 16] = 12.0
        for i in range(1, 16):
            r[b * 16 + i] = 2 * mids[(b + i) % 7] * (-1) ** (i + b)
    rows.append(r)
    # bf16 neighbours of the ties
    r2 = r.copy()
    bits = torch.from_numpy(r2).to(torch.bfloat16).view(torch.int16)
    bits[1::3] += 1
    bits[2::3] -= 1
    rows.append(bits.view(torch.bfloat16).float().numpy())
    # zeros, negative zeros, one non-zero
    r3 = np.zeros(k, np.float32)
    r3[1::2] = -0.0
    r3[100] = 1.0
    rows.append(r3)
    # subnormal bf16 values and tiny blocks
    rows.append((np.random.default_rng(1).standard_normal(k) * 1e-39).astype(np.float32))
    # huge values
    rows.append((np.random.default_rng(2).standard_normal(k) * 1e30).astype(np.float32))
    # powers of two and (6, 8) x 2^e saturation for MX
    r6 = np.tile(np.array([4.0, 7.0, -7.5, 6.0, 0.5, 1.0, 2.0, 3.0], np.float32), k // 8)
    rows.append(r6)
    return torch.from_numpy(np.stack(rows)).to(torch.bfloat16)


@pytest.mark.parametrize("fmt,mode,st", [(0, 0, 0.0), (0, 1, 1.0), (1, 0, 0.0)])
def test_adversarial(F, O, fmt, mode, st):
    check_quant(F, O, _adversarial(), fmt, mode, st)


def _every_bf16_magnitude(rows, seed):
    """Rows of 4096: every bf16 value of magnitude in [2^-8, 2^8) with both
    signs, each row a seeded permutation (so blocks mix binades)."""
    mags = ((1.0 + np.arange(128)[None, :] / 128.0) * 2.0 ** np.arange(-8, 8)[:, None]).ravel()
    vals = np.concatenate([mags, -mags]).astype(np.float32)  # 8 significant bits: exact in bf16
    rng = np.random.default_rng(seed)
    return torch.from_numpy(np.stack([rng.permutation(vals) for _ in range(rows)])).to(torch.bfloat16)


@pytest.mark.parametrize("part", range(4))
def test_nvfp4_global_scale_sweep(F, O, part):
    """Global scales A / 2688 for every bf16 significand A, as a static scale
    and as the dynamic scale of a tensor whose abs-max is A: the divisors
    d = s_b s_g of some of these put E2M1 midpoints times d on bf16 values
    (the codes then come from the bracket or from divisions), the rest take
    the one-multiply path.  Every code and scale byte must match the oracle."""
    x = _every_bf16_magnitude(4, part)
    for a in range(part * 32, part * 32 + 32):
        amax = 256.0 + 2.0 * a  # a bf16 value above every element of x
        check_quant(F, O, x, 0, mode=1, st=float(np.float32(amax / 2688.0)))
        xd = x.clone()
        xd[a % 4, (a * 37) % 4096] = -amax
        check_quant(F, O, xd, 0)


def test_all_zero_tensor(F, O):
    x = torch.zeros((5, 256), dtype=torch.bfloat16)
    check_quant(F, O, x, 0)
    check_quant(F, O, x, 1)
    c, s, g = gpu_quant(F, x, 0)
    assert g == 0.0 and not c.any() and not s.any()


def test_negative_zero_code(F, O):
    """A negative value that rounds to zero keeps its sign (code 0x8): the
    oracle's reading, checked against the device conversion."""
    x = torch.tensor([[6.0, -0.01] + [0.0] * 30], dtype=torch.bfloat16)
    c, s, g = gpu_quant(F, x, 0, 1, 1.0)
    assert c[0, 0] == 0x87
    check_quant(F, O, x, 0, 1, 1.0)


def test_zero_rows_is_noop(F):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q = F.quantize(x, 0)
    torch.cuda.synchronize()
    assert q.codes.numel() == 0


@pytest.mark.parametrize("rows,k,fmt", [(8192, 4096, 0), (2048, 7168, 1)])
def test_full_size_activations(F, O, rows, k, fmt):
    """The prefill (NVFP4) and MXFP4 workloads' activations, every element."""
    check_quant(F, O, I.randn_bf16((rows, k), 2 if fmt == 0 else 4), fmt)


def test_weight_prepack_full_size(F, O):
    w = I.weights_bf16(14336, 4096, 102)
    q = F.prepack_weight(w.cuda())
    torch.cuda.synchronize()
    c_o, s_o, g_o = O.quantize_nvfp4(I.u16(w))
    assert np.array_equal(q.codes.cpu().numpy(), c_o)
    assert np.array_equal(q.scales.cpu().numpy(), O.scales_to_mma(s_o, 14336, 4096, 0))
    assert np.float32(q.gscale.cpu()[0]) == np.float32(g_o)
