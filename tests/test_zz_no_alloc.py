"""fp4_quantize_act_noalloc: the quantiser entry point that takes no
workspace, for callers that cannot allocate device memory (its amax scratch
is a static device array inside the library).  Called through the C ABI and
compared with fp4_quantize_act (which takes a workspace) bit for bit, on two
calls in a row so that the second call runs on the scratch the first one
left behind.  This file is collected last on purpose."""
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


def _noalloc(F, x, fmt, mode=0, st=0.0):
    rows, k = x.shape
    q = F.empty_qtensor(fmt, rows, k, x.device)
    F._check(F.lib().fp4_quantize_act_noalloc(fmt, F._ptr(x), rows, k, mode, float(st), F._ptr(q.codes),
                                              F._ptr(q.scales), F._ptr(q.gscale), F._stream()))
    return q


def _same(a, b):
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes)
    assert torch.equal(a.scales, b.scales)
    assert a.gscale.cpu().numpy().tobytes() == b.gscale.cpu().numpy().tobytes()


@pytest.mark.parametrize("fmt,mode,st", [(0, 0, 0.0), (1, 0, 0.0), (0, 1, 0.02)])
def test_noalloc_matches_workspace_entry_point(F, fmt, mode, st):
    # two calls in a row with different inputs and sizes
    for shape, seed in [((300, 1024), 11), ((4096, 4096), 12)]:
        x = I.randn_bf16(shape, seed).cuda()
        if seed == 12:
            x[7, 9] = 40.0  # move the tensor amax so a stale partial would show
        got = _noalloc(F, x, fmt, mode, st)
        ref = F.quantize(x, fmt, mode, st)
        _same(got, ref)
    F.device_status()


def test_noalloc_rejects_bad_arguments(F):
    L = F.lib()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    q = F.empty_qtensor(0, 4, 64, "cuda")
    st = L.fp4_quantize_act_noalloc(0, F._ptr(x), 4, 48, 0, 0.0, F._ptr(q.codes), F._ptr(q.scales),
                                    F._ptr(q.gscale), F._stream())
    assert st == F.STATUS_CODE["FP4_ERR_SHAPE"]
    st = L.fp4_quantize_act_noalloc(0, F._ptr(x), 4, 64, 1, 0.0, F._ptr(q.codes), F._ptr(q.scales),
                                    F._ptr(q.gscale), F._stream())
    assert st == F.STATUS_CODE["FP4_ERR_INVALID_SCALE"]
