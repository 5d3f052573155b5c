"""The fp32 block-update GEMM (tensor cores with 3 x TF32 products, or FFMA) against a
float64 product, through the C ABI test helper gptq_gemm_f32."""
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


def _run(g, M, N, K, ak, bk, engine, alpha=1.0, beta=0.0, lower=False, seed=0):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    Ad = torch.from_numpy(np.ascontiguousarray(A if ak else A.T)).cuda()
    Bd = torch.from_numpy(np.ascontiguousarray(B.T if bk else B)).cuda()
    Cd = torch.from_numpy(C0.copy()).cuda()
    g.gptq_gemm_f32(Ad, Bd, Cd, ak, bk, alpha=alpha, beta=beta, engine=engine, lower_tiles=lower)
    torch.cuda.synchronize()
    ref = beta * C0.astype(np.float64) + alpha * (A.astype(np.float64) @ B.astype(np.float64))
    got = Cd.cpu().numpy().astype(np.float64)
    if lower:
        I = np.arange(M)[:, None] // 128
        J = np.arange(N)[None, :] // 128
        keep = J <= I
        assert np.array_equal(got[~keep], C0.astype(np.float64)[~keep]), "tiles above the diagonal must stay"
        got, ref = got[keep], ref[keep]
    # elementwise: |error| <= c * K * 2^-21 * sum_k |a_ik b_kj| (+ the rounding of C)
    scale = np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64) + np.abs(beta * C0)
    if lower:
        scale = scale[keep]
    return np.max(np.abs(got - ref) / scale)


@pytest.mark.parametrize("engine", [0, 1])
@pytest.mark.parametrize("ak,bk", [(True, True), (True, False), (False, True), (False, False)])
def test_gemm_layouts(g, engine, ak, bk):
    err = _run(g, 300, 260, 200, ak, bk, engine, alpha=-1.0, beta=1.0)
    assert err < 4.0 * 2.0 ** -21, err


@pytest.mark.parametrize("engine", [0, 1])
def test_gemm_lower_tiles_and_ragged(g, engine):
    err = _run(g, 384, 384, 64, True, True, engine, alpha=-1.0, beta=1.0, lower=True, seed=3)
    assert err < 4.0 * 2.0 ** -21, err
    err = _run(g, 129, 257, 33, True, True, engine, alpha=0.5, beta=0.0, seed=4)
    assert err < 4.0 * 2.0 ** -21, err


def test_gemm_long_k_accuracy(g):
    """K = 4096: partial products are summed in fp32 registers per 32-deep chunk, so the
    tensor-core result stays within a few units of fp32 rounding of the FFMA one."""
    e_tc = _run(g, 256, 256, 4096, True, True, 0, seed=5)
    e_ff = _run(g, 256, 256, 4096, True, True, 1, seed=5)
    assert e_tc < 4.0 * 2.0 ** -21 and e_ff < 2.0 ** -21, (e_tc, e_ff)
