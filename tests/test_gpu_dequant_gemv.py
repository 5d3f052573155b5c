"""gptq_dequant_gemv: Y = X W_hat^T straight from the packed layer, against the oracle's
dequantize-and-multiply in float64 on the GPU's own quantized output (codes, scales,
zeros and, for act-order groups, g_idx)."""
import numpy as np
import pytest
import torch

from oracle import gptq_oracle as orc
from synth import ActSpec, bf16_bits_to_f32, make_activations, make_weight

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from post_weight_quantization_gb300 import build as b
    b.build()
    from post_weight_quantization_gb300 import gptq
    return gptq


def _g_idx(perm, d, gs):
    gi = np.empty(d, dtype=np.int64)
    gi[perm] = np.arange(d) // (d if gs == -1 else gs)
    return gi


def _check(g, q, m, d, bits, gs, perm, T, seed, rows=None):
    gi = None if perm is None else _g_idx(perm.cpu().numpy().astype(np.int64), d, gs)
    gi_dev = None if gi is None else torch.from_numpy(gi.astype(np.int32)).cuda()
    Xb = make_activations(ActSpec("heavy_tail", T, d, seed=seed))
    Xd = torch.from_numpy(Xb.view(np.int16)).cuda()
    Y = g.gptq_dequant_gemv(q, Xd, m, g_idx=gi_dev)
    torch.cuda.synchronize()
    g.gptq_device_check()
    words = q.qweight.cpu().numpy().view(np.uint32)
    sc, ze = q.scales.cpu().numpy(), q.zeros.cpu().numpy()
    if rows is not None:
        words, sc, ze = words[rows], sc[rows], ze[rows]
    X = bf16_bits_to_f32(Xb).astype(np.float64)
    ref = orc.dequant_matmul(X, words, sc, ze, bits, gs, gi)
    What = orc.dequantize_packed(words, sc, ze, bits, d, gs, gi)
    bound = (d + 2) * 2.0 ** -24 * (np.abs(X) @ np.abs(What).T) + 1e-30
    got = Y.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[:, rows]
    assert got.shape == ref.shape
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


@pytest.mark.parametrize("bits,gs,ao", [(4, 128, False), (3, -1, True), (2, 64, True), (8, 32, False),
                                        (4, 128, True)])
@pytest.mark.parametrize("T", [1, 5, 11])
def test_dequant_gemv_matches_oracle(g, bits, gs, ao, T):
    m, d = 200, 768
    W_bits = make_weight(m, d, 51)
    X_bits = make_activations(ActSpec("heavy_tail", 4096, d, seed=51))
    Wd = torch.from_numpy(W_bits.view(np.int16)).cuda().view(torch.bfloat16)
    q, _, _, perm = g.quantize_layer(Wd, [torch.from_numpy(X_bits.view(np.int16)).cuda()], bits=bits, group_size=gs,
                                     blocksize=32 if gs == 32 else 64, act_order=ao)
    _check(g, q, m, d, bits, gs, perm, T, seed=100 + T)


def test_dequant_gemv_full_size_layer(g):
    """The 4096 x 4096 4-bit g128 layer (Hessian from 16384 tokens), eight tokens,
    sampled rows against the oracle."""
    m = d = 4096
    W_bits = make_weight(m, d, 1)
    X_bits = make_activations(ActSpec("heavy_tail", 16384, d, seed=1))
    Wd = torch.from_numpy(W_bits.view(np.int16)).cuda().view(torch.bfloat16)
    q, _, _, _ = g.quantize_layer(Wd, [torch.from_numpy(X_bits.view(np.int16)).cuda()], bits=4, group_size=128)
    rows = np.sort(np.random.default_rng(3).choice(m, size=96, replace=False))
    _check(g, q, m, d, 4, 128, None, 8, seed=7, rows=rows)
