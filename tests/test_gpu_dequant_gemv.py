"""gptq_dequant_gemv: Y = X W_hat^T straight from a packed layer, against the oracle's
dequantize-and-multiply in float64.

The packed layers are built on the CPU from seeded random codes, zeros and scales (and,
for act-order groups, a random column order giving g_idx) and packed by the oracle's
bitstream packer, so both sides read the same bytes and nothing the oracle consumes
comes from the GPU."""
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


def packed_layer(m, d, bits, gs, act_order, seed):
    rng = np.random.default_rng(seed)
    G = 1 if gs == -1 else d // gs
    codes = rng.integers(0, 2 ** bits, size=(m, d))
    zeros = rng.integers(0, 2 ** bits, size=(m, G)).astype(np.float32)
    scales = (0.002 * (0.5 + rng.random((m, G)))).astype(np.float32)
    gi = None
    if act_order and G > 1:
        perm = rng.permutation(d)
        gi = np.empty(d, dtype=np.int64)
        gi[perm] = np.arange(d) // gs           # groups formed in processing order
    return orc.pack_codes(codes, bits), scales, zeros, gi


def _check(g, m, d, bits, gs, act_order, T, seed, rows=None):
    words, sc, ze, gi = packed_layer(m, d, bits, gs, act_order, seed)
    q = g.QuantizedLayer(torch.from_numpy(words.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                         torch.from_numpy(ze).cuda(), torch.zeros(d, device="cuda"), bits, gs, d)
    gi_dev = None if gi is None else torch.from_numpy(gi.astype(np.int32)).cuda()
    Xb = make_activations(ActSpec("heavy_tail", T, d, seed=seed + 1))
    Xd = torch.from_numpy(Xb.view(np.int16)).cuda()
    Y = g.gptq_dequant_gemv(q, Xd, m, g_idx=gi_dev)
    torch.cuda.synchronize()
    g.gptq_device_check()
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


# Codes in natural groups run on the tensor cores (one, two or four units of a row per
# thread and block: g32, g64 and g128 at 4 bits, g64, g128 and per-channel at 2 bits;
# three-word units at 3 bits, g128, g256 and per-channel; two-word units at 8 bits,
# g32, g128 and per-channel); act-order groups (g_idx) and groups narrower than a
# block (2-bit g32, 3-bit g64) on the FMA kernel. m = 200 leaves a partial 16-row
# tile; T = 11 is a piece of eight and one of three tokens.
@pytest.mark.parametrize("bits,gs,ao", [(4, 128, False), (3, -1, True), (2, 64, True), (8, 32, False),
                                        (4, 128, True), (4, 64, False), (4, 32, False), (4, -1, False),
                                        (2, 64, False), (2, 128, False), (2, -1, True), (2, 32, False),
                                        (3, 128, False), (3, 256, False), (3, 64, False), (3, 128, True),
                                        (8, 128, False), (8, -1, False), (8, 64, True)])
@pytest.mark.parametrize("T", [1, 5, 11])
def test_dequant_gemv_matches_oracle(g, bits, gs, ao, T):
    _check(g, 200, 768, bits, gs, ao, T, seed=100 + T + bits)


@pytest.mark.parametrize("bits,gs", [(4, 128), (2, 64), (3, -1), (8, 128)])
def test_dequant_gemv_full_size_layer(g, bits, gs):
    """A 4096 x 4096 packed layer (4-bit g128, 2-bit g64, 3-bit per-channel, 8-bit g128),
    eight tokens, sampled rows against the oracle."""
    rows = np.sort(np.random.default_rng(3).choice(4096, size=96, replace=False))
    _check(g, 4096, 4096, bits, gs, False, 8, seed=7, rows=rows)
