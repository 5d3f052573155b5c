"""GPU parity on the method's degenerate cases, through the whole path (Hessian product,
factor and column loop) or the column loop alone, against what the pages fix:

  * a diagonal Hessian: every off-diagonal entry of Hinv1 is an exact zero, so no
    column moves and GPTQ is round-to-nearest with the same quantizer ("GPTQ: fixing
    errors as you go", the OBQ update with zero off-diagonals); codes, scales and
    zeros must equal the oracle's round-to-nearest bit for bit, in natural order and
    with act-order (groups formed in processing order);
  * a degenerate group (max == min): the listing of "GPTQ-style round-to-nearest with
    Hessian weighting" clamps the scale to 1e-8 and lets the codes clamp; constant
    rows of zeros, of a positive and of a negative value;
  * exact round-half-even ties, built from dyadic weights whose scale is a power of
    two: the codes and the zero point must come out as hand-computed.

A diagonal Hessian comes from calibration tokens that each touch one channel only.
"""
import numpy as np
import pytest
import torch

from oracle import gptq_oracle as orc
from synth import bf16_bits_to_f32, make_weight
from synth.workloads import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    from post_weight_quantization_gb300 import build as b
    b.build()
    from post_weight_quantization_gb300 import gptq
    return gptq


def dev_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def one_channel_tokens(d: int, reps: int = 2) -> np.ndarray:
    """reps * d tokens; token t carries a value on channel t % d only, so X^T X is
    diagonal. Channel c's values are bf16(1 + c / 64) with alternating signs: many
    channels share a diagonal value exactly (bf16 rounding), which exercises the
    act-order tie rule as well."""
    n = reps * d
    X = np.zeros((n, d), dtype=np.float32)
    t = np.arange(n)
    c = t % d
    X[t, c] = (1.0 + c / 64.0).astype(np.float32) * np.where((t // d) % 2 == 0, 1.0, -1.0)
    return f32_to_bf16_bits(X)


def gpu_path(g, W_bits, X_bits, bits, gs, act_order):
    m, d = W_bits.shape
    Wd = dev_bits(W_bits).view(torch.bfloat16)
    q, H, U, perm = g.quantize_layer(Wd, [dev_bits(X_bits)], bits=bits, group_size=gs, blocksize=128,
                                     act_order=act_order)
    torch.cuda.synchronize()
    g.gptq_device_check()
    codes = g.gptq_unpack_codes(q.qweight, m, d, bits).cpu().numpy().astype(np.int64)
    return q, codes, U, perm


def rtn_f32(W32, bits, gs, perm=None):
    """The oracle's round-to-nearest in float32 (the listing's precision), in processing
    order when a permutation is given, returned in the original column order."""
    Wp = W32 if perm is None else W32[:, perm]
    r = orc.rtn(np.ascontiguousarray(Wp, dtype=np.float32), bits, gs, dtype=np.float32)
    codes = r["codes"]
    if perm is not None:
        codes = np.empty_like(r["codes"])
        codes[:, perm] = r["codes"]
    return codes, r["scales"], r["zeros"]


@pytest.mark.parametrize("bits,gs,act_order", [(4, 128, False), (2, 64, False), (3, -1, True), (4, 128, True),
                                               (8, 32, False)])
def test_diagonal_hessian_is_round_to_nearest(g, bits, gs, act_order):
    m, d = 200, 512
    W_bits = make_weight(m, d, 5)
    W32 = bf16_bits_to_f32(W_bits)
    # constant groups in some rows: stay constant (nothing moves with a diagonal H)
    g_eff = d if gs == -1 else gs
    W32[3, :] = 0.0
    W32[7, g_eff:2 * g_eff if g_eff < d else d] = 0.0125
    W32[11, :g_eff] = -0.03125
    W_bits = f32_to_bf16_bits(W32)
    W32 = bf16_bits_to_f32(W_bits)
    X_bits = one_channel_tokens(d)
    q, codes, U, perm = gpu_path(g, W_bits, X_bits, bits, gs, act_order)
    Ug = U.cpu().numpy()
    assert np.count_nonzero(Ug - np.diag(np.diag(Ug))) == 0, "Hinv1 of a diagonal H must be diagonal"
    po = None
    if act_order:
        po = orc.act_order_perm(orc.hessian([bf16_bits_to_f32(X_bits)]))
        assert np.array_equal(perm.cpu().numpy(), po)
    c_ref, s_ref, z_ref = rtn_f32(W32, bits, gs, po)
    assert np.array_equal(codes, c_ref)
    assert np.array_equal(q.scales.cpu().numpy(), s_ref)
    assert np.array_equal(q.zeros.cpu().numpy(), z_ref)


def test_degenerate_groups_in_one_block_match_float32_oracle(g):
    """Constant rows with a general Hessian: the first group's max == min, so its scale is
    clamped to 1e-8 and its codes clamp; one block is bit-identical to the float32
    oracle."""
    m, d, bits, gs = 64, 128, 4, 128
    rng = np.random.default_rng(3)
    W32 = bf16_bits_to_f32(make_weight(m, d, 9))
    W32[0, :] = 0.0
    W32[1, :] = 0.015625
    W32[2, :] = -0.25
    W32[5, :] = 3.0e-3
    W32 = bf16_bits_to_f32(f32_to_bf16_bits(W32))
    X = rng.standard_normal((1024, d)).astype(np.float32)
    H = orc.hessian([bf16_bits_to_f32(f32_to_bf16_bits(X))])
    Hd, _ = orc.damp(H, 0.01)
    U32 = orc.hinv1(Hd).astype(np.float32)
    res = orc.gptq_columns(W32, U32, bits, gs, 128, dtype=np.float32)
    q = g.gptq_quantize_layer(torch.from_numpy(W32).cuda(), torch.from_numpy(U32).cuda(), bits=bits, group_size=gs,
                              blocksize=128, sync=True)
    codes = g.gptq_unpack_codes(q.qweight, m, d, bits).cpu().numpy().astype(np.int64)
    sc, ze = q.scales.cpu().numpy(), q.zeros.cpu().numpy()
    assert np.array_equal(codes, res["codes"])
    assert np.array_equal(sc, res["scales"]) and np.array_equal(ze, res["zeros"])
    # the degenerate rows: scale clamped to 1e-8, zero and codes clamped
    assert np.all(sc[[0, 1, 2, 5], 0] == np.float32(1e-8))
    assert ze[1, 0] == 0 and ze[2, 0] == 15 and ze[5, 0] == 0
    assert codes[1, 0] == 15 and codes[2, 0] == 0 and codes[0, 0] == 0


def test_round_half_even_ties_are_hand_computed(g):
    """Dyadic weights with a power-of-two scale put w / scale + zero exactly on .5 ties
    (4-bit, groups of 32, diagonal Hessian so nothing moves):
      row 0: min = -7/64, max = 8/64 -> scale 1/64, zero 7; w = (k + 1/2)/64 gives
             k + 7.5, rounded to the even neighbour;
      row 1: min = -7.5/64, max = 7.5/64 -> scale 1/64 and -min/scale = 7.5 exactly,
             so the zero point itself rounds half to even (8)."""
    d, bits, gs = 128, 4, 32
    ks = np.arange(-7, 8)                                     # 15 tie values per group
    W = np.zeros((2, d), dtype=np.float64)
    for grp in range(d // gs):
        base = grp * gs
        row0 = np.concatenate([[-7.0, 8.0], ks + 0.5, np.full(gs - 2 - len(ks), 1.0)]) / 64.0
        row1 = np.concatenate([[-7.5, 7.5], ks + 0.5, np.full(gs - 2 - len(ks), 0.0)]) / 64.0
        W[0, base:base + gs] = row0
        W[1, base:base + gs] = row1
    W32 = W.astype(np.float32)
    W_bits = f32_to_bf16_bits(W32)
    assert np.array_equal(bf16_bits_to_f32(W_bits), W32), "the tie weights must be exact in bf16"
    q, codes, _, _ = gpu_path(g, W_bits, one_channel_tokens(d), bits, gs, False)
    sc, ze = q.scales.cpu().numpy(), q.zeros.cpu().numpy()
    assert np.all(sc == np.float32(1 / 64))
    assert np.all(ze[0] == 7) and np.all(ze[1] == 8)
    for grp in range(d // gs):
        base = grp * gs
        tie0 = codes[0, base + 2: base + 2 + len(ks)]
        tie1 = codes[1, base + 2: base + 2 + len(ks)]
        exp0 = [(k + 7) if (k + 7) % 2 == 0 else (k + 8) for k in ks]       # k + 7.5 to even
        exp1 = [min(15, (k + 8) if (k + 8) % 2 == 0 else (k + 9)) for k in ks]  # k + 8.5 to even
        assert tie0.tolist() == exp0, (grp, tie0.tolist(), exp0)
        assert tie1.tolist() == exp1, (grp, tie1.tolist(), exp1)
        assert codes[0, base] == 0 and codes[0, base + 1] == 15              # min and max
        assert codes[1, base] == 0 and codes[1, base + 1] == 15              # -7.5+8 = 0.5 -> 0; 15.5 -> 15
