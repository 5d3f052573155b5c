"""gptq_dequant_gemm: Y = X W_hat^T on the tensor cores straight from a packed layer,
against the oracle's dequantize-and-multiply in float64.

The packed layers are built on the CPU from seeded random codes, zeros and scales and
packed by the oracle's bitstream packer (pinned against hand-packed words), so both
sides read the same bytes and nothing the oracle consumes comes from the GPU.

Tolerance: every product X[t][j] (code - zero) is exact in fp32 and each group's
partial sum is formed in fp32, then scaled and added in fp32, so
|Y - Y64| <= (unit + G + 2) 2^-23 sum_j |X[t][j]| |w_hat[r][j]| with `unit` the columns
summed in one tensor-memory accumulator (at most 256) and G the groups per row. bf16
output: within that bound plus half a bf16 unit in the last place of |Y64|, and equal to
the fp32 output rounded to nearest even.
"""
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


def packed_layer(m, d, bits, gs, seed):
    """Seeded random codes, integer zeros and positive scales, packed by the oracle."""
    rng = np.random.default_rng(seed)
    G = 1 if gs == -1 else d // gs
    codes = rng.integers(0, 2 ** bits, size=(m, d))
    zeros = rng.integers(0, 2 ** bits, size=(m, G)).astype(np.float32)
    scales = (0.002 * (0.5 + rng.random((m, G)))).astype(np.float32)
    words = orc.pack_codes(codes, bits)
    return words, scales, zeros


def unit_of(d, gs):
    g_ = d if gs == -1 else gs
    u = g_
    if u > 256:
        u = 256
        while g_ % u:
            u //= 2
    return u


def run_gemm(g, words, scales, zeros, m, d, bits, gs, Xb, out_bf16):
    q = g.QuantizedLayer(torch.from_numpy(words.view(np.int32)).cuda(), torch.from_numpy(scales).cuda(),
                         torch.from_numpy(zeros).cuda(), torch.zeros(d, device="cuda"), bits, gs, d)
    Y = g.gptq_dequant_gemm(q, torch.from_numpy(Xb.view(np.int16)).cuda(), m, out_bf16=out_bf16)
    torch.cuda.synchronize()
    g.gptq_device_check()
    return Y


@pytest.mark.parametrize("m,d,T,bits,gs", [(256, 512, 384, 4, 128), (200, 768, 300, 3, -1), (130, 256, 129, 2, 64),
                                           (96, 512, 1000, 8, 32), (384, 1024, 256, 4, 256), (64, 96, 77, 4, 32),
                                           (160, 4096, 512, 4, 128), (128, 640, 200, 2, 64)])
def test_dequant_gemm_matches_oracle(g, m, d, T, bits, gs):
    words, scales, zeros = packed_layer(m, d, bits, gs, seed=m + d + bits)
    Xb = make_activations(ActSpec("heavy_tail", T, d, seed=T + d))
    X = bf16_bits_to_f32(Xb).astype(np.float64)
    ref = orc.dequant_matmul(X, words, scales, zeros, bits, gs)
    What = orc.dequantize_packed(words, scales, zeros, bits, d, gs)
    G = 1 if gs == -1 else d // gs
    bound = (unit_of(d, gs) + G + 2) * 2.0 ** -23 * (np.abs(X) @ np.abs(What).T) + 1e-30
    Y = run_gemm(g, words, scales, zeros, m, d, bits, gs, Xb, False).cpu().numpy().astype(np.float64)
    assert Y.shape == ref.shape
    assert np.all(np.abs(Y - ref) <= bound), float(np.max(np.abs(Y - ref) / bound))
    Yb = run_gemm(g, words, scales, zeros, m, d, bits, gs, Xb, True)
    # the bf16 output is the fp32 output rounded to nearest even
    assert torch.equal(Yb, torch.from_numpy(Y.astype(np.float32)).cuda().to(torch.bfloat16))
    yb = Yb.float().cpu().numpy().astype(np.float64)
    half_ulp = np.abs(ref) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(yb - ref) <= bound + half_ulp)


def test_dequant_gemm_llama_layer_sampled(g):
    """The 4096 x 4096 4-bit g128 layer on 16384 tokens in one call (128 token tiles x 32
    row tiles, every CTA persistent over many tiles), sampled tokens against float64."""
    m = d = 4096
    T = 16384
    words, scales, zeros = packed_layer(m, d, 4, 128, seed=11)
    Xb = make_activations(ActSpec("heavy_tail", T, d, seed=12))
    Y = run_gemm(g, words, scales, zeros, m, d, 4, 128, Xb, False)
    toks = np.sort(np.random.default_rng(4).choice(T, size=64, replace=False))
    X = bf16_bits_to_f32(Xb[toks]).astype(np.float64)
    ref = orc.dequant_matmul(X, words, scales, zeros, 4, 128)
    What = orc.dequantize_packed(words, scales, zeros, 4, d, 128)
    bound = (128 + 32 + 2) * 2.0 ** -23 * (np.abs(X) @ np.abs(What).T)
    got = Y.cpu().numpy()[toks].astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


def test_dequant_gemm_argument_errors(g):
    words, scales, zeros = packed_layer(64, 256, 4, 128, seed=1)
    Xb = make_activations(ActSpec("heavy_tail", 16, 256, seed=1))
    q = g.QuantizedLayer(torch.from_numpy(words.view(np.int32)).cuda(), torch.from_numpy(scales).cuda(),
                         torch.from_numpy(zeros).cuda(), torch.zeros(256, device="cuda"), 4, 128, 256)
    X = torch.from_numpy(Xb.view(np.int16)).cuda()
    before = g.gptq_launch_count()
    with pytest.raises(ValueError):
        g.gptq_dequant_gemm(q, X, 64, ws=torch.empty(10, dtype=torch.uint8, device="cuda"))
    lib = g.library()
    st = lib.gptq_dequant_gemm(q.qweight.data_ptr(), q.scales.data_ptr(), q.zeros.data_ptr(), 64, 250, 4, 128,
                               X.data_ptr(), 16, 256, X.data_ptr(), 0, 64, X.data_ptr(), 1 << 20, None)
    assert st == g.GPTQ_ERR_INVALID_ARG
    assert g.gptq_launch_count() == before
