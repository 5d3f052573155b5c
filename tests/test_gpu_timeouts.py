"""A bounded on-device wait that runs out. Every spin-wait in the library gives up after a
wall-clock limit, raises the device error word and returns with nothing in flight, so
the context stays usable. The library's own wait routines run here on something that
never completes (a counter nothing publishes; an mbarrier nothing arrives on) with a
1 ms limit; nothing faults, traps or hangs."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from post_weight_quantization_gb300 import build as b
    b.build()
    from post_weight_quantization_gb300 import gptq
    return gptq


@pytest.mark.parametrize("which", [0, 1])
def test_wait_gives_up_and_reports_timeout(g, which):
    g.gptq_device_check()                                  # start from a clear error word
    st = g.gptq_wait_selftest(which, limit_ns=1_000_000)
    assert st == g.GPTQ_ERR_TIMEOUT, g.gptq_status_string(st)
    assert "gave up" in g.gptq_last_error()
    with pytest.raises(g.GPTQError) as ei:
        g.gptq_device_check()
    assert ei.value.status == g.GPTQ_ERR_TIMEOUT
    g.gptq_device_check()                                  # read once, then cleared


def test_context_still_usable_after_a_timeout(g):
    assert g.gptq_wait_selftest(1, limit_ns=1_000_000) == g.GPTQ_ERR_TIMEOUT
    with pytest.raises(g.GPTQError):
        g.gptq_device_check()
    # a small layer still quantizes normally afterwards
    W = torch.randn((64, 128), device="cuda") * 0.02
    X = (torch.randn((512, 128), device="cuda")).to(torch.bfloat16)
    q, H, U, _ = g.quantize_layer(W, [X], bits=4, group_size=128, blocksize=128)
    torch.cuda.synchronize()
    g.gptq_device_check()
    codes = g.gptq_unpack_codes(q.qweight, 64, 128, 4).cpu().numpy()
    assert codes.max() <= 15 and np.isfinite(q.scales.cpu().numpy()).all()
