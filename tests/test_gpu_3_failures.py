"""Failure detection without a GPU fault: a device-side wait on a barrier
that nothing completes must give up after its limit, report
FP4_ERR_DEVICE_TIMEOUT through fp4_device_status, and leave the context
usable for the next call."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__ as ge
    ge.build()
    from mxfp4_block_scaled_gb300 import fp4
    return fp4


def test_bounded_wait_reports_timeout(F):
    L = F.lib()
    F.device_status()  # clean slate
    F._check(L.fp4_debug_timeout_probe(2000, F._stream()))
    assert L.fp4_device_status(F._stream()) == F.STATUS_CODE["FP4_ERR_DEVICE_TIMEOUT"]
    assert "gave up" in L.fp4_last_error_message().decode()
    # flag cleared, context still usable
    assert L.fp4_device_status(F._stream()) == 0
    x = torch.randn(64, 256, device="cuda").to(torch.bfloat16)
    q = F.quantize(x)
    torch.cuda.synchronize()
    assert q.gscale.item() > 0


def test_unsupported_arch_status_on_device(F):
    L = F.lib()
    x = torch.randn(16, 64, device="cuda").to(torch.bfloat16)
    L.fp4_set_arch_override(90)
    try:
        with pytest.raises(F.FP4Error) as e:
            F.quantize(x)
        assert e.value.name == "FP4_ERR_UNSUPPORTED_ARCH"
    finally:
        L.fp4_set_arch_override(0)
    F.quantize(x)
    torch.cuda.synchronize()
