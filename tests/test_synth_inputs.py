"""The seeded input generators shared by the oracle and the CUDA path (CPU): bf16
rounding, determinism across threads and chunk ranges, the stated statistics of the
recipes, and the workload shapes."""
import numpy as np
import pytest

from synth import ActSpec, bf16_bits_to_f32, make_activations, make_weight
from synth.workloads import CHUNK, f32_to_bf16_bits, gen_activations_into, workload


def test_bf16_rounding_is_nearest_even():
    one = np.float32(1.0)
    ulp = np.float32(2.0 ** -7)                    # bf16 spacing just above 1
    x = np.array([1.0, one + ulp / 2, one + ulp + ulp / 2, one + ulp / 4, one + 3 * ulp / 4, -2.5, 0.0, -0.0],
                 dtype=np.float32)
    got = bf16_bits_to_f32(f32_to_bf16_bits(x))
    want = np.array([1.0, 1.0, one + 2 * ulp, 1.0, one + ulp, -2.5, 0.0, -0.0], dtype=np.float32)
    assert np.array_equal(got, want)
    assert np.signbit(got[-1])
    # every bf16 value is a fixed point, and widening is exact
    b = np.arange(0, 1 << 16, 97, dtype=np.uint32).astype(np.uint16)
    f = bf16_bits_to_f32(b)
    finite = np.isfinite(f)
    assert np.array_equal(f32_to_bf16_bits(f[finite]), b[finite])


@pytest.mark.parametrize("kind", ["heavy_tail", "gauss_cov", "silu_gate"])
def test_activations_do_not_depend_on_threads_or_ranges(kind):
    spec = ActSpec(kind, 3 * CHUNK + 100, 96, seed=5)
    a = make_activations(spec, threads=1)
    b = make_activations(spec, threads=4)
    assert np.array_equal(a, b)
    part = np.empty((CHUNK, 96), dtype=np.uint16)
    gen_activations_into(spec, part, threads=2, token_range=(CHUNK, 2 * CHUNK))
    assert np.array_equal(part, a[CHUNK:2 * CHUNK])
    with pytest.raises(ValueError):
        gen_activations_into(spec, part, token_range=(1, CHUNK + 1))


def test_weights_are_seeded_normal():
    w1 = make_weight(2048, 64, seed=9, layer=2, threads=1)
    w2 = make_weight(2048, 64, seed=9, layer=2, threads=3)
    assert np.array_equal(w1, w2)
    assert not np.array_equal(w1, make_weight(2048, 64, seed=9, layer=3))
    w = bf16_bits_to_f32(w1).astype(np.float64)
    assert abs(w.mean()) < 5e-4 and abs(w.std() - 0.02) < 5e-4


def test_heavy_tail_recipe_statistics():
    """X = (T_z M)/8 + 0.5 T_e with unit-variance Student-t(4) entries, 1 % of the
    channels scaled x30: plain channels have variance 64/64 + 0.25 = 1.25 in
    expectation over M, outlier channels 900 times that, and the tails are heavy."""
    d = 400
    X = bf16_bits_to_f32(make_activations(ActSpec("heavy_tail", 2 * CHUNK, d, seed=2))).astype(np.float64)
    var = X.var(axis=0)
    out = var > 100.0
    assert out.sum() == round(0.01 * d)
    assert 0.7 < np.median(var[~out]) < 2.0
    assert 300.0 < np.median(var[out] / np.median(var[~out])) < 2000.0
    e = X[:, ~out] - X[:, ~out].mean(axis=0)
    kurt = np.mean(e ** 4, axis=0) / np.mean(e ** 2, axis=0) ** 2
    assert np.median(kurt) > 3.5                        # Gaussian: 3
    # low-rank mixing correlates channels: |cov| ~ |N(0, 1/64)|, so the median |corr| is
    # about 0.67 / 8 / 1.25 = 0.067, against about 0.007 for independent channels here
    c = np.corrcoef(X[:, ~out][:, :50].T)
    assert np.median(np.abs(c[np.triu_indices(50, 1)])) > 0.04


def test_workload_shapes():
    wl = workload("llama_4096_g128")
    assert [(l.m, l.d) for l in wl.layers] == [(4096, 4096)]
    assert wl.acts["in"].n == 128 * 2048 and (wl.bits, wl.group_size, wl.blocksize) == (4, 128, 128)
    wl = workload("llama_4096_3bit_actorder")
    assert (wl.bits, wl.group_size, wl.act_order) == (3, -1, True)
    wl = workload("llama7b_mlp")
    assert [(l.m, l.d) for l in wl.layers] == [(11008, 4096), (11008, 4096), (4096, 11008)]
    assert {k: (a.n, a.d) for k, a in wl.acts.items()} == {"mlp_in": (262144, 4096), "mlp_down": (262144, 11008)}
    wl = workload("llama70b_block")
    assert [(l.name, l.m, l.d) for l in wl.layers] == [
        ("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
        ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)]
    assert all(a.n == 131072 for a in wl.acts.values())
    wl = workload("toy_256")
    assert [(l.m, l.d) for l in wl.layers] == [(256, 256)] and wl.acts["in"].n == 512
