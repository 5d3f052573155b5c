"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests compares the oracle with itself or retypes its formulas: each
checks a closed form, an invariant the pages state, an exact-arithmetic restatement
of a different formulation, a brute-force search, or a hand-worked fixture under
tests/golden/.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import gptq_oracle as orc
from synth import ActSpec, bf16_bits_to_f32, make_activations, make_weight
from synth.workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _layer(m, d, n, seed, kind="heavy_tail", outliers=None):
    W = bf16_bits_to_f32(make_weight(m, d, seed)).astype(np.float64)
    X = bf16_bits_to_f32(make_activations(ActSpec(kind, n, d, seed=seed, outlier_count=outliers)))
    return W, X.astype(np.float64)


@pytest.fixture(scope="module")
def toy():
    """The 256 x 256 toy layer (512 Gaussian correlated tokens, 4 outlier channels x20)."""
    W = bf16_bits_to_f32(make_weight(256, 256, 0)).astype(np.float64)
    X = bf16_bits_to_f32(make_activations(
        ActSpec("gauss_cov", 512, 256, seed=0, outlier_count=4, outlier_scale=20.0))).astype(np.float64)
    return W, X, orc.hessian([X])


# ----------------------------------------------------------------------------------
# quantizer
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_quantizer_is_nearest_level(bits):
    """clamp(round(w/s + z)) must be the nearest of all 2^b grid levels (exhaustive)."""
    rng = np.random.default_rng(bits)
    wg = rng.normal(0, 0.02, size=(64, 32))
    s, z = orc.quant_params(wg, bits)
    w = rng.normal(0, 0.03, size=(64, 200))          # includes values outside [min, max]
    q = orc.quantize(w, s[:, None], z[:, None], bits)
    levels = np.arange(2 ** bits)
    vals = (levels[None, None, :] - z[:, None, None]) * s[:, None, None]
    best = np.argmin(np.abs(w[:, :, None] - vals), axis=2)
    assert np.array_equal(q.astype(np.int64), best)
    assert q.min() >= 0 and q.max() <= 2 ** bits - 1


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_quant_params_span_the_group(bits):
    """Level 0 and level 2^b-1 land within s/2 of the group's min and max; zero is an
    integer in range; inside [min, max] dequantized values are within s/2."""
    rng = np.random.default_rng(10 + bits)
    wg = rng.normal(0, 0.02, size=(128, 128))
    s, z = orc.quant_params(wg, bits)
    qmax = 2 ** bits - 1
    assert np.all(z == np.round(z)) and z.min() >= 0 and z.max() <= qmax
    inner = (z > 0) & (z < qmax)
    assert inner.any()
    assert np.all(np.abs(-z * s - wg.min(1))[inner] <= s[inner] / 2 + 1e-15)
    assert np.all(np.abs((qmax - z) * s - wg.max(1))[inner] <= s[inner] / 2 + 1e-15)
    q = orc.quantize(wg, s[:, None], z[:, None], bits)
    wq = orc.dequantize(q, s[:, None], z[:, None])
    assert np.all(np.abs(wq - wg)[inner] <= (s[:, None] / 2 + 1e-15)[inner])


def test_degenerate_group_clamps():
    """max == min: scale is clamped to 1e-8 and the codes clamp into range."""
    wg = np.full((3, 8), 0.25)
    s, z = orc.quant_params(wg, 4)
    assert np.all(s == 1e-8)
    assert np.all(z == 0)
    q = orc.quantize(wg, s[:, None], z[:, None], 4)
    assert np.all(q == 15)


# ----------------------------------------------------------------------------------
# damping, act-order, Cholesky chain (golden fixtures and closed forms)
# ----------------------------------------------------------------------------------
def test_damping_golden():
    g = _golden("damping_actorder.json")
    for case in g["damping"]:
        H = np.array(case["H"], dtype=np.float64)
        Hd, lam = orc.damp(H, case["percdamp"])
        assert lam == pytest.approx(case["lambda"], rel=1e-15)
        assert np.allclose(np.diag(Hd), case["diag_damped"], rtol=1e-15)
        off = ~np.eye(len(H), dtype=bool)
        assert np.array_equal(Hd[off], H[off])


def test_damping_rejects_nonpositive():
    with pytest.raises(ValueError):
        orc.damp(np.zeros((3, 3)), 0.01)


def test_act_order_golden():
    for case in _golden("damping_actorder.json")["act_order"]:
        H = np.diag(np.array(case["diag"], dtype=np.float64))
        assert orc.act_order_perm(H).tolist() == case["perm"]


def test_hinv1_golden_2x2():
    for case in _golden("hinv1_2x2.json")["cases"]:
        U = orc.hinv1(np.array(case["H_d"], dtype=np.float64))
        assert np.allclose(U, case["U"], rtol=1e-14, atol=1e-15)


def test_hinv1_diagonal_closed_form():
    h = np.array([1.0, 4.0, 0.25, 9.0, 2.0])
    U = orc.hinv1(np.diag(h))
    assert np.allclose(U, np.diag(1 / np.sqrt(h)), rtol=1e-15, atol=0)


def test_hinv1_properties(toy):
    """U upper with positive diagonal and U^T U H_d = I (residual ~ kappa * eps)."""
    _, _, H = toy
    Hd, _ = orc.damp(H, 0.01)
    U = orc.hinv1(Hd)
    assert np.allclose(np.tril(U, -1), 0)
    assert np.all(np.diag(U) > 0)
    kappa = np.linalg.cond(Hd)
    assert np.abs(U.T @ U @ Hd - np.eye(len(Hd))).max() < 50 * kappa * np.finfo(float).eps


def test_hinv1_reverse_identity(toy):
    """Hinv1 = J chol_lower(J H_d J)^-1 J (J the reversal): the same factor by a
    different route (uniqueness of the Cholesky factor with positive diagonal)."""
    _, _, H = toy
    Hd, _ = orc.damp(H, 0.01)
    J = np.eye(len(Hd))[::-1]
    L = np.linalg.cholesky(J @ Hd @ J)
    U2 = J @ np.linalg.inv(L) @ J
    U = orc.hinv1(Hd)
    assert np.abs(U - U2).max() <= 1e-10 * np.abs(U).max()


# ----------------------------------------------------------------------------------
# Hessian
# ----------------------------------------------------------------------------------
def test_hessian_is_the_objectives_quadratic_form():
    """||dW X^T||_F^2 == 1/2 tr(dW H dW^T) for H = 2 X^T X: pins the factor 2 and the
    orientation (objective and Hessian of 'GPTQ: fixing errors as you go')."""
    rng = np.random.default_rng(3)
    X = rng.normal(size=(300, 40))
    dW = rng.normal(size=(7, 40))
    H = orc.hessian([X])
    direct = np.sum((dW @ X.T) ** 2)
    assert orc.loss_quadratic_form(dW, H) == pytest.approx(direct, rel=1e-12)


def test_hessian_streaming_and_integers():
    """Accumulating over batches equals one pass; integer data gives exact integers."""
    rng = np.random.default_rng(4)
    X = rng.integers(-8, 9, size=(1000, 24)).astype(np.float64)
    H1 = orc.hessian([X])
    H2 = orc.hessian([X[:333], X[333:700], X[700:]])
    assert np.array_equal(H1, H2)
    assert np.array_equal(H1, np.round(H1))
    # one token: 2 x x^T has rank one and diagonal 2 x_i^2
    x = X[:1]
    H = orc.hessian([x])
    assert np.linalg.matrix_rank(H) == 1
    assert np.array_equal(np.diag(H), 2 * x[0] ** 2)
    # sampled entries agree with the full product
    rows, cols = np.array([0, 3, 23]), np.array([5, 3, 0])
    assert np.array_equal(orc.hessian_entries(X, rows, cols), H1[rows, cols])


# ----------------------------------------------------------------------------------
# exact-rational OBQ in fixed order ("GPTQ: fixing errors as you go", The OBQ update)
# ----------------------------------------------------------------------------------
def _frac_inverse(A):
    n = len(A)
    M = [list(row) + [Fraction(int(i == j)) for j in range(n)] for i, row in enumerate(A)]
    for c in range(n):
        p = next(r for r in range(c, n) if M[r][c] != 0)
        M[c], M[p] = M[p], M[c]
        piv = M[c][c]
        M[c] = [v / piv for v in M[c]]
        for r in range(n):
            if r != c and M[r][c] != 0:
                f = M[r][c]
                M[r] = [a - f * b for a, b in zip(M[r], M[c])]
    return [row[n:] for row in M]


def _frac_quant(wg, bits):
    qmax = 2 ** bits - 1
    mn, mx = min(wg), max(wg)
    s = (mx - mn) / qmax
    if s < Fraction(1e-8):
        s = Fraction(1e-8)
    z = min(max(round(-mn / s), 0), qmax)
    return s, Fraction(z)


def _obq_fixed_order(w0, Hd, bits, g):
    """One row: quantize columns 0..d-1 in order; after each, update the free weights
    by delta_F = -(w_q - quant(w_q)) / [H_F^-1]_qq * (H_F^-1)_{:,q} and remove q from
    H_F^-1 by one step of Gaussian elimination. Exact rationals throughout."""
    d = len(w0)
    Hi = _frac_inverse(Hd)
    w = list(w0)
    free = list(range(d))
    codes, losses, scales = [], [], []
    qmax = 2 ** bits - 1
    for q in range(d):
        if q % g == 0:
            s, z = _frac_quant(w[q:q + g], bits)
            scales.append((s, z))
        c = min(max(round(w[q] / s + z), 0), qmax)
        wq = (c - z) * s
        r = w[q] - wq
        hqq = Hi[q][q]
        codes.append(c)
        losses.append(r * r / (2 * hqq))
        for k in free:
            w[k] -= r / hqq * Hi[k][q]
        free.remove(q)
        col = [Hi[a][q] for a in range(d)]
        rowq = list(Hi[q])
        for a in free:
            for b in free:
                Hi[a][b] -= col[a] * rowq[b] / hqq
    return codes, losses, scales


@pytest.mark.parametrize("bits,g,bs", [(2, 3, 1), (2, 3, 3), (3, 2, 4), (3, -1, 2), (4, 6, 6), (2, 2, 6)])
def test_oracle_equals_exact_obq(bits, g, bs):
    """The Cholesky-row form (Hinv1 rows, blocked) equals the explicit OBQ downdate form
    in exact arithmetic: identical codes, scales and per-element losses."""
    rng = np.random.default_rng(100 + bits * 10 + bs)
    m, d = 3, 6
    X = rng.integers(-3, 4, size=(5, d)).astype(np.float64)   # rank-deficient: damping needed
    W = rng.integers(-200, 201, size=(m, d)) / 1024.0
    H = orc.hessian([X])
    Hd, _ = orc.damp(H, 0.01)
    U = orc.hinv1(Hd)
    res = orc.gptq_columns(W, U, bits, g, bs)
    gg = d if g == -1 else g
    Hd_f = [[Fraction(v) for v in row] for row in Hd]
    for r in range(m):
        codes, losses, scales = _obq_fixed_order([Fraction(v) for v in W[r]], Hd_f, bits, gg)
        assert res["codes"][r].tolist() == codes
        np.testing.assert_allclose(res["losses"][r], [float(x) for x in losses], rtol=1e-9, atol=1e-18)
        np.testing.assert_allclose(res["scales"][r], [float(s) for s, _ in scales], rtol=1e-12)
        np.testing.assert_array_equal(res["zeros"][r], [float(z) for _, z in scales])


# ----------------------------------------------------------------------------------
# blocking, special cases and brute force
# ----------------------------------------------------------------------------------
def test_blocksize_does_not_change_codes(toy):
    """'GPTQ, Line by Line': the blocksize does not change the result (fp64 codes identical
    for blocksize 1, 32, 128 and d; P3's unblocked listing is blocksize 1)."""
    W, _, H = toy
    Hd, _ = orc.damp(H, 0.01)
    U = orc.hinv1(Hd)
    ref = orc.gptq_columns(W, U, 4, 128, 1)
    for bs in (32, 128, 256):
        res = orc.gptq_columns(W, U, 4, 128, bs)
        assert np.array_equal(res["codes"], ref["codes"])
        assert np.array_equal(res["zeros"], ref["zeros"])
        np.testing.assert_allclose(res["scales"], ref["scales"], rtol=1e-12)
        np.testing.assert_allclose(res["losses"], ref["losses"], rtol=1e-8, atol=1e-20)


def test_blocksize_invariance_per_channel_act_order():
    """Same invariance for 3-bit per-channel act-order (blocksize 32 vs 128 vs 1)."""
    W, X = _layer(48, 256, 1024, seed=7)
    H = orc.hessian([X])
    a = orc.gptq_layer(W, H, 3, -1, 32, act_order=True)
    b = orc.gptq_layer(W, H, 3, -1, 128, act_order=True)
    c = orc.gptq_layer(W, H, 3, -1, 1, act_order=True)
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["codes"], c["codes"])


def test_diagonal_hessian_is_rtn():
    """With a diagonal H every off-diagonal Hinv1 entry is zero, so no compensation
    happens and GPTQ reduces to round-to-nearest, bit for bit."""
    rng = np.random.default_rng(5)
    W = rng.normal(0, 0.02, size=(32, 256))
    H = np.diag(rng.uniform(0.5, 3.0, size=256))
    for g, bs in ((128, 128), (64, 128), (-1, 32)):
        res = orc.gptq_layer(W, H, 4, g, bs)
        ref = orc.rtn(W, 4, g)
        assert np.array_equal(res["codes"], ref["codes"])
        assert np.array_equal(res["W_hat"], ref["W_hat"])


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_single_column_is_exhaustive_optimum(bits):
    """d = 1: GPTQ = RTN = the best of all 2^b codes for the quadratic loss."""
    rng = np.random.default_rng(bits)
    W = rng.normal(0, 0.02, size=(20, 1))
    H = np.array([[2.5]])
    res = orc.gptq_layer(W, H, bits, -1, 1)
    # with one column the group has min == max: the clamp gives scale 1e-8 -> code clamps;
    # use the scale/zero GPTQ chose and search all codes
    s, z = res["scales"][:, 0], res["zeros"][:, 0]
    levels = (np.arange(2 ** bits)[None, :] - z[:, None]) * s[:, None]
    loss = 0.5 * (W - levels) ** 2 * (H[0, 0] + res["lambda"])
    assert np.array_equal(res["codes"][:, 0], np.argmin(loss, axis=1))
    assert np.array_equal(res["codes"], orc.rtn(W, bits, -1)["codes"])


def _ls_free_optimum(w0, Hd, fixed_idx, fixed_val):
    """argmin over the free coordinates of 1/2 (w - w0) Hd (w - w0)^T with w fixed on
    fixed_idx: w_F = w0_F - Hd_FF^-1 Hd_FX (v - w0_X)."""
    d = len(w0)
    Fi = [k for k in range(d) if k not in set(fixed_idx)]
    w = w0.copy()
    if fixed_idx:
        dv = np.asarray(fixed_val) - w0[fixed_idx]
        w[Fi] = w0[Fi] - np.linalg.solve(Hd[np.ix_(Fi, Fi)], Hd[np.ix_(Fi, fixed_idx)] @ dv)
        w[fixed_idx] = fixed_val
    return w


def test_each_step_is_the_obq_choice():
    """At every step the code GPTQ takes is the best of all 2^b candidates when the
    columns to its right are re-optimized by least squares (the OBQ step), and GPTQ's
    group statistics are taken from those least-squares-optimal weights."""
    rng = np.random.default_rng(11)
    m, d, bits, g = 4, 6, 2, 3
    X = rng.normal(size=(40, d)) @ rng.normal(size=(d, d))
    W = rng.normal(0, 0.02, size=(m, d))
    H = orc.hessian([X])
    res = orc.gptq_layer(W, H, bits, g, 3)
    Hd = res["H_d"]
    for r in range(m):
        for j in range(d):
            prev = list(range(j))
            vals = list(res["W_hat"][r, :j])
            wopt = _ls_free_optimum(W[r], Hd, prev, vals)
            s, z = res["scales"][r, j // g], res["zeros"][r, j // g]
            if j % g == 0:
                grp = wopt[j:j + g]
                assert s == pytest.approx((grp.max() - grp.min()) / (2 ** bits - 1), rel=1e-9)
            best, best_loss = None, np.inf
            for c in range(2 ** bits):
                w = _ls_free_optimum(W[r], Hd, prev + [j], vals + [(c - z) * s])
                loss = orc.loss_quadratic_form((w - W[r])[None, :], Hd)
                if loss < best_loss - 1e-18:
                    best, best_loss = c, loss
            assert res["codes"][r, j] == best


def test_exhaustive_search_lower_bounds_gptq():
    """GPTQ is greedy: the best of all (2^b)^d code vectors (same scales and zeros) never
    loses to it, and the loss identity makes both comparable."""
    rng = np.random.default_rng(12)
    d, bits = 5, 2
    X = rng.normal(size=(30, d)) @ rng.normal(size=(d, d))
    W = rng.normal(0, 0.02, size=(3, d))
    H = orc.hessian([X])
    res = orc.gptq_layer(W, H, bits, -1, d)
    Hd = res["H_d"]
    for r in range(3):
        s, z = res["scales"][r, 0], res["zeros"][r, 0]
        best = min(orc.loss_quadratic_form(((np.array(c) - z) * s - W[r])[None, :], Hd)
                   for c in itertools.product(range(2 ** bits), repeat=d))
        gptq = orc.loss_quadratic_form((res["W_hat"][r] - W[r])[None, :], Hd)
        assert best <= gptq * (1 + 1e-12)
        assert res["losses"][r].sum() == pytest.approx(gptq, rel=1e-10)


def test_loss_identity(toy):
    """Sum of Losses1 = 1/2 tr(dW H_d dW^T) = ||dW X^T||^2 + lambda/2 ||dW||^2."""
    W, X, H = toy
    res = orc.gptq_layer(W, H, 4, 128, 128)
    dW = W - res["W_hat"]
    total = res["losses"].sum()
    assert total == pytest.approx(orc.loss_quadratic_form(dW, res["H_d"]), rel=1e-10)
    direct = np.sum((dW @ X.T) ** 2) + 0.5 * res["lambda"] * np.sum(dW ** 2)
    assert total == pytest.approx(direct, rel=1e-9)


def test_hessian_scale_by_four(toy):
    """H -> 4H: lambda x4, Hinv1 x1/2, errors x2, updates unchanged: identical codes,
    scales and zeros; losses x4 exactly (powers of two)."""
    W, _, H = toy
    a = orc.gptq_layer(W, H, 4, 128, 128)
    b = orc.gptq_layer(W, 4 * H, 4, 128, 128)
    assert np.array_equal(a["codes"], b["codes"])
    assert np.array_equal(a["scales"], b["scales"]) and np.array_equal(a["zeros"], b["zeros"])
    np.testing.assert_allclose(b["losses"], 4 * a["losses"], rtol=1e-12, atol=0)


def test_act_order_is_permutation_equivariant():
    """act-order output = the natural-order loop on permuted W and H, scattered back."""
    W, X = _layer(40, 128, 600, seed=8)
    H = orc.hessian([X])
    res = orc.gptq_layer(W, H, 3, -1, 32, act_order=True)
    p = res["perm"]
    assert np.all(np.diff(np.diag(H)[p]) <= 0)
    Hd, _ = orc.damp(H, 0.01)
    U = orc.hinv1(Hd[np.ix_(p, p)])
    nat = orc.gptq_columns(W[:, p], U, 3, -1, 32)
    assert np.array_equal(res["codes"][:, p], nat["codes"])
    assert np.array_equal(res["losses"][:, p], nat["losses"])


def test_rows_are_independent(toy):
    W, _, H = toy
    full = orc.gptq_layer(W, H, 4, 128, 128)
    top = orc.gptq_layer(W[:100], H, 4, 128, 128)
    bot = orc.gptq_layer(W[100:], H, 4, 128, 128)
    assert np.array_equal(full["codes"], np.vstack([top["codes"], bot["codes"]]))
    assert np.array_equal(full["scales"], np.vstack([top["scales"], bot["scales"]]))


def test_gptq_beats_rtn_on_correlated_inputs(toy):
    """'GPTQ: fixing errors as you go': the compensation lowers the output error."""
    W, _, H = toy
    res = orc.gptq_layer(W, H, 4, 128, 128)
    e_gptq = orc.relative_output_error(W, res["W_hat"], H)
    e_rtn = orc.relative_output_error(W, orc.rtn(W, 4, 128)["W_hat"], H)
    assert e_gptq < 0.8 * e_rtn


@pytest.mark.parametrize("n,ao", [(333, False), (333, True), (40, True)])
def test_relative_output_error_is_the_direct_output_norm(n, ao):
    """The output error through H equals ||(W - W_hat) X^T||_F / ||W X^T||_F computed from
    the tokens themselves ("GPTQ: fixing errors as you go", Objective: the error of the
    layer's outputs on the calibration inputs). Non-square W and X, more and fewer
    tokens than channels (a singular H), and an act-order result in original column
    order; a missing square root, the damped instead of the plain Hessian, or a
    transposed product would each fail."""
    m, d = 48, 96
    W, X = _layer(m, d, n, seed=21 + n)
    H = orc.hessian([X])                                  # 2 X^T X, undamped
    res = orc.gptq_layer(W, H, 3, 32, 32, 0.01, act_order=ao)
    direct = np.linalg.norm((W - res["W_hat"]) @ X.T) / np.linalg.norm(W @ X.T)
    assert 1e-4 < direct < 1.0
    got = orc.relative_output_error(W, res["W_hat"], H)
    assert abs(got - direct) <= 1e-12 * direct, (got, direct)
    # any positive multiple of X^T X gives the same ratio (H / n, as one listing keeps it)
    assert abs(orc.relative_output_error(W, res["W_hat"], H / (7.0 * n)) - direct) <= 1e-12 * direct
    # the damped Hessian gives a different (larger) number: the metric uses the plain one
    Hd, _ = orc.damp(H, 0.01)
    assert orc.relative_output_error(W, res["W_hat"], Hd) > direct * (1 + 1e-6)


def test_codes_in_range_all_bits(toy):
    W, _, H = toy
    for bits, g in ((2, 64), (3, -1), (4, 128), (8, 128)):
        res = orc.gptq_layer(W, H, bits, g, 128)
        assert res["codes"].min() >= 0 and res["codes"].max() <= 2 ** bits - 1
        assert np.all(res["zeros"] == np.round(res["zeros"]))


def test_rejects_bad_grouping():
    W = np.zeros((2, 192))
    U = np.eye(192)
    with pytest.raises(ValueError):
        orc.gptq_columns(W, U, 4, 96, 128)     # neither divides the other
    with pytest.raises(ValueError):
        orc.gptq_columns(W, U, 4, 128, 128)    # 192 % 128 != 0


# ----------------------------------------------------------------------------------
# packing
# ----------------------------------------------------------------------------------
def test_pack_golden():
    for case in _golden("pack_codes.json")["cases"]:
        codes = np.array([case["codes"]])
        words = orc.pack_codes(codes, case["bits"])
        assert [f"0x{w:08x}" for w in words[0]] == case["words"]
        assert np.array_equal(orc.unpack_codes(words, case["bits"], codes.shape[1]), codes)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_pack_roundtrip(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(5, 263))
    words = orc.pack_codes(codes, bits)
    assert words.shape == (5, (263 * bits + 31) // 32)
    assert np.array_equal(orc.unpack_codes(words, bits, 263), codes)


# ----------------------------------------------------------------------------------
# act-order with groups: groups are formed in processing order
# ----------------------------------------------------------------------------------
def test_act_order_groups_diagonal_hessian_is_rtn_in_processing_order():
    """Diagonal H with distinct entries: no compensation, so act-order with groups is
    round-to-nearest applied to the columns in processing order (groups of g
    consecutive processed columns), scattered back; g_idx maps each column to its group."""
    rng = np.random.default_rng(17)
    d, g = 256, 64
    W = rng.normal(0, 0.02, size=(24, d))
    H = np.diag(rng.permutation(np.linspace(0.5, 3.0, d)))
    res = orc.gptq_layer(W, H, 4, g, 128, act_order=True)
    p = res["perm"]
    assert not np.array_equal(p, np.arange(d))
    ref = orc.rtn(W[:, p], 4, g)
    assert np.array_equal(res["codes"][:, p], ref["codes"])
    assert np.array_equal(res["scales"], ref["scales"]) and np.array_equal(res["zeros"], ref["zeros"])
    inv = np.empty(d, dtype=np.int64)
    inv[p] = np.arange(d)
    assert np.array_equal(res["g_idx"], inv // g)
    gi = res["g_idx"]
    np.testing.assert_array_equal(res["W_hat"], (res["codes"] - res["zeros"][:, gi]) * res["scales"][:, gi])


def test_act_order_groups_with_equal_diagonal_is_the_natural_order():
    """Equal diagonal entries (H[i][j] = rho^|i-j|): the stable act-order sort keeps the
    natural order, so act-order with groups gives the grouped natural-order result."""
    d = 256
    i = np.arange(d)
    H = 0.7 ** np.abs(i[:, None] - i[None, :])
    W = np.random.default_rng(3).normal(0, 0.02, size=(20, d))
    a = orc.gptq_layer(W, H, 4, 128, 128, act_order=True)
    b = orc.gptq_layer(W, H, 4, 128, 128)
    assert np.array_equal(a["perm"], np.arange(d))
    for k in ("codes", "scales", "zeros", "W_hat", "losses"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(a["g_idx"], np.arange(d) // 128)


def test_act_order_groups_blocksize_invariance():
    """The pages' blocksize invariance holds with act-order and groups (identical fp64
    codes for blocksize 1, 32 and 128)."""
    W, X = _layer(24, 256, 600, seed=12)
    H = orc.hessian([X])
    r = [orc.gptq_layer(W, H, 4, 64, bs, act_order=True) for bs in (1, 32, 128)]
    assert not np.array_equal(r[0]["perm"], np.arange(256))
    for x in r[1:]:
        assert np.array_equal(x["codes"], r[0]["codes"])
        np.testing.assert_allclose(x["scales"], r[0]["scales"], rtol=1e-12)


# ----------------------------------------------------------------------------------
# the stored layer used again: dequantize and multiply
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("bits,gs,ao", [(4, 128, False), (3, -1, True), (2, 64, True), (8, 32, False)])
def test_dequantize_packed_reproduces_w_hat(bits, gs, ao):
    """The packed codes with the group scales and zeros (g_idx for act-order) give back
    exactly the W_hat the quantizer produced, and Y = X W_hat^T follows from it."""
    W, X = _layer(12, 256, 512, seed=bits + 7)
    H = orc.hessian([X])
    res = orc.gptq_layer(W, H, bits, gs, 32 if gs == 32 else 64, act_order=ao)
    words = orc.pack_codes(res["codes"], bits)
    What = orc.dequantize_packed(words, res["scales"], res["zeros"], bits, 256, gs, res["g_idx"] if ao else None)
    assert np.array_equal(What, res["W_hat"])
    Xt = X[:5]
    np.testing.assert_allclose(orc.dequant_matmul(Xt, words, res["scales"], res["zeros"], bits, gs,
                                                  res["g_idx"] if ao else None), Xt @ res["W_hat"].T, rtol=1e-12)


# ----------------------------------------------------------------------------------
# layers one after another
# ----------------------------------------------------------------------------------
def _bf16_table():
    """Every finite positive bfloat16 value, ascending, with its bit pattern."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    return bf16_bits_to_f32(bits).astype(np.float64), bits


def test_round_to_bf16_is_nearest_with_ties_to_even():
    """Brute force over the whole bfloat16 table: each result is a bfloat16 value, no
    other one is nearer, and exact midpoints go to the neighbour with an even last
    mantissa bit. For float32 inputs it also agrees with the input generators' bit-level
    float32 rounding, a different construction."""
    vals, bits = _bf16_table()
    rng = np.random.default_rng(21)
    y = rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000))
    k = rng.integers(200, len(vals) - 200, 500)
    mids = 0.5 * (vals[k] + vals[k + 1])                  # exact in float64
    y = np.concatenate([y, mids, -mids, vals[k], [0.0]])
    r = orc.round_to_bf16(y)
    a = np.abs(y)
    i = np.clip(np.searchsorted(vals, a), 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]
    dlo, dhi = a - lo, hi - a
    want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(bits[i - 1] % 2 == 0, lo, hi)))
    want = np.where(a == 0, 0.0, np.copysign(want, y))
    assert np.array_equal(r, want)
    assert np.all(np.abs(r[len(y) - 1 - 3 * 500:len(y) - 1 - 500]) != 0)
    x32 = (rng.standard_normal(20000) * np.exp(rng.uniform(-40, 40, 20000))).astype(np.float32)
    assert np.array_equal(orc.round_to_bf16(x32.astype(np.float64)),
                          bf16_bits_to_f32(f32_to_bf16_bits(x32)).astype(np.float64))


@pytest.mark.parametrize("ao,gs", [(False, 16), (True, 16), (True, -1)])
def test_sequential_pass_second_hessian_is_the_quantized_sandwich(ao, gs):
    """Kept in float64 between layers, X_2 = X_1 W_hat_1^T, so H_2 = W_hat_1 H_1 W_hat_1^T:
    the quantized weights (not the original ones), in the original column order (act-order
    undone) and the right orientation, carry the inputs onward."""
    W1 = bf16_bits_to_f32(make_weight(48, 64, seed=4, layer=0)).astype(np.float64)
    W2 = bf16_bits_to_f32(make_weight(32, 48, seed=4, layer=1)).astype(np.float64)
    X = bf16_bits_to_f32(make_activations(ActSpec("heavy_tail", 600, 64, seed=4))).astype(np.float64)
    res = orc.sequential_pass(X, [W1, W2], bits=3, group_size=gs, blocksize=16, act_order=ao, propagate=None)
    H1, H2 = res["H"]
    Wh = res["layers"][0]["W_hat"]
    want = Wh @ H1 @ Wh.T
    np.testing.assert_allclose(H2, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())
    assert not np.allclose(H2, W1 @ H1 @ W1.T, rtol=1e-3)
    # the second layer is quantized against that Hessian
    assert res["layers"][1]["codes"].shape == (32, 48)


def _on_grid_weight(m, d, bits, g, rng):
    """W = (code - zero) * scale with every row of every group holding the codes 0 and
    2^b - 1 and a power-of-two scale: min/max give back exactly that scale and zero."""
    q = rng.integers(0, 2 ** bits, size=(m, d))
    q[:, 0::g] = 0
    q[:, 1::g] = 2 ** bits - 1
    z = rng.integers(0, 2 ** bits, size=(m, d // g)).astype(np.float64)
    s = np.ldexp(1.0, -rng.integers(5, 9, size=(m, d // g)))
    gi = np.arange(d) // g
    return (q - z[:, gi]) * s[:, gi], q, s, z


def test_sequential_pass_on_grid_weights_is_the_plain_product_chain():
    """Weights already on their grid quantize to themselves with zero error, so nothing is
    compensated and the pass reduces to X_0 W_1^T W_2^T W_3^T exactly; with bfloat16 between
    layers every recorded input is a bfloat16 value within half an ulp of the float chain's."""
    rng = np.random.default_rng(8)
    X0 = bf16_bits_to_f32(make_activations(ActSpec("gauss_cov", 300, 64, seed=8))).astype(np.float64)
    shapes = [(96, 64), (64, 96), (32, 64)]
    Ws, Qs = [], []
    for m, d in shapes:
        W, q, s, z = _on_grid_weight(m, d, 4, 32, rng)
        Ws.append(W)
        Qs.append((q, s, z))
    res = orc.sequential_pass(X0, Ws, bits=4, group_size=32, blocksize=32, propagate=None)
    for lay, W, (q, s, z) in zip(res["layers"], Ws, Qs):
        assert np.array_equal(lay["codes"], q)
        assert np.array_equal(lay["scales"], s) and np.array_equal(lay["zeros"], z)
        assert np.array_equal(lay["W_hat"], W)
        assert np.all(lay["losses"] == 0)
    assert np.array_equal(res["output"], X0 @ Ws[0].T @ Ws[1].T @ Ws[2].T)
    rb = orc.sequential_pass(X0, Ws, bits=4, group_size=32, blocksize=32)
    chain = X0 @ Ws[0].T
    x1 = rb["inputs"][1]
    assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(x1.astype(np.float32))).astype(np.float64), x1)
    assert np.all(np.abs(x1 - chain) <= np.ldexp(np.abs(chain), -8))   # 8 significant bits


def test_sequential_pass_layers_are_the_single_layer_path_on_their_inputs():
    """Every layer of the pass is the single-layer path on H = 2 X_l^T X_l of the inputs it
    records (bfloat16 values: the Hessian sees the rounded inputs, as a Hessian built from
    stored bfloat16 activations does); a chain whose widths do not meet is refused."""
    W, X = _layer(16, 64, 256, seed=30)
    W2 = bf16_bits_to_f32(make_weight(24, 16, seed=30, layer=1)).astype(np.float64)
    res = orc.sequential_pass(X, [W, W2], bits=4, group_size=16, blocksize=16)
    for Wl, Xl, lay in zip((W, W2), res["inputs"], res["layers"]):
        ref = orc.gptq_layer(Wl, 2.0 * (Xl.T @ Xl), 4, 16, 16)
        for k in ("codes", "scales", "zeros", "W_hat", "losses"):
            assert np.array_equal(lay[k], ref[k]), k
    x1 = res["inputs"][1]
    assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(x1.astype(np.float32))).astype(np.float64), x1)
    with pytest.raises(ValueError):
        orc.sequential_pass(X, [W, np.zeros((8, 15))], bits=4, group_size=-1, blocksize=16)
