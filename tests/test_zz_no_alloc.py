"""gptq_factor_static: the factor for callers that cannot allocate device memory
(a runtime that owns the GPU's memory through its own pool, or a pipeline that
cannot take cudaMalloc's implicit synchronization). Its scratch is a device array
inside the library, so the test checks that two calls in a row, through the C ABI,
give what the workspace entry point gives on the same inputs, and that sizes beyond
the array are refused before anything runs.

This file is collected last so that a run stopping at the first failure has run
every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import gptq_oracle as orc
from synth import ActSpec, bf16_bits_to_f32, make_activations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from post_weight_quantization_gb300 import build as b
    b.build()
    from post_weight_quantization_gb300 import gptq
    return gptq


def _hessian(d, n, seed):
    X = bf16_bits_to_f32(make_activations(ActSpec("heavy_tail", n, d, seed=seed))).astype(np.float64)
    return orc.hessian([X]).astype(np.float32)


def _static_call(g, H, d, act_order):
    """Direct C-ABI call of gptq_factor_static (no binding helper)."""
    U = torch.empty((d, d), dtype=torch.float32, device="cuda")
    perm = torch.empty(d, dtype=torch.int32, device="cuda")
    info = ctypes.c_int64(-7)
    st = g.library().gptq_factor_static(H.data_ptr(), d, ctypes.c_float(0.01), int(act_order),
                                        perm.data_ptr() if act_order else None, U.data_ptr(), ctypes.byref(info),
                                        torch.cuda.current_stream().cuda_stream)
    assert st == g.GPTQ_OK, g.gptq_last_error()
    assert info.value == -1
    return U, (perm if act_order else None)


def test_static_factor_matches_workspace_factor_twice(g):
    """Two calls in a row on different inputs (the second must not see the first's
    scratch). Both entry points run the same kernels in the same order on the same
    inputs, so Hinv1 must agree bit for bit; the oracle's chain bounds both."""
    for d, n, seed, act_order in ((2048, 8192, 11, False), (768, 4096, 12, True)):
        Hn = _hessian(d, n, seed)
        H = torch.from_numpy(Hn).cuda()
        U_s, p_s = _static_call(g, H, d, act_order)
        U_w, p_w, info = g.gptq_factor(H, percdamp=0.01, act_order=act_order)
        torch.cuda.synchronize()
        assert info == -1
        if act_order:
            assert torch.equal(p_s, p_w)
        assert torch.equal(U_s, U_w), "static-scratch factor differs from the workspace factor"
        Hd, _ = orc.damp(Hn.astype(np.float64), 0.01)
        perm = orc.act_order_perm(Hn.astype(np.float64)) if act_order else np.arange(d)
        Uo = orc.hinv1(Hd[np.ix_(perm, perm)])
        kappa = np.linalg.cond(Hd)
        a = U_s.cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(a - Uo) / np.linalg.norm(Uo)
        assert rel < 50 * kappa * 2.0 ** -24, (rel, kappa)
    g.gptq_device_check()


def test_static_factor_refuses_sizes_beyond_its_scratch(g):
    before = g.gptq_launch_count()
    info = ctypes.c_int64(0)
    P = 0x10000000   # never dereferenced: the size check comes first
    st = g.library().gptq_factor_static(P, 2049, ctypes.c_float(0.01), 0, None, P, ctypes.byref(info), None)
    assert st == g.GPTQ_ERR_INVALID_ARG
    assert "2048" in g.gptq_last_error()
    assert g.gptq_launch_count() == before
