"""The per-stage bounds bench.py reports, against hand-derived figures (CPU)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6788.6, "bf16_tflops": 1917.0, "sm_max_mhz": 2070.0}


def test_llama_4096_g128_bounds():
    r = bench.stage_rooflines(4096, 4096, 262144, 4, 128, 128, syrk_ms=2.68, quantize_ms=1.25, peaks=PEAKS)
    q = r["column_loop_and_lazy_update"]
    # W in bf16 + upper triangle of Hinv1 + 4-bit codes + scales and zeros + column losses
    assert q["bytes"] == 2 * 4096 ** 2 + 2 * 4096 * 4097 + 4096 ** 2 // 2 + 8 * 4096 * 32 + 4 * 4096 == 76570624
    # lazy updates: block b (of 32) updates the 128 * (31 - b) columns right of it
    assert q["flops_lazy"] == 2 * 4096 * 128 * 128 * sum(range(32))
    # rank-one updates inside a block: column t moves the 127 - t columns after it
    assert q["flops_in_block"] == 32 * 2 * 4096 * sum(127 - t for t in range(128))
    p_tf32 = 1917e12 * 1.1 / 2.25
    p_ffma = 152 * 128 * 2 * 2070e6
    t1 = q["flops_lazy"] / p_tf32 + q["flops_in_block"] / p_ffma
    assert q["bound_ms"] == pytest.approx(t1 * 1e3, abs=1e-4)
    assert q["bound_ms_three_pass"] == pytest.approx((2 * q["flops_lazy"] / p_tf32 + t1) * 1e3, abs=1e-4)
    assert q["frac"] == pytest.approx(q["bound_ms"] / 1.25, abs=1e-4)
    s = r["syrk"]
    assert s["bound_ms"] == pytest.approx(262144 * 4096 * 4097 / 1917e12 * 1e3, abs=1e-4)
    assert s["frac"] == pytest.approx(s["bound_ms"] / 2.68, abs=1e-4)
    assert "factor" not in r
    f = bench.stage_rooflines(4096, 4096, 262144, 4, 128, 128, 2.68, 1.25, PEAKS, factor_ms=1.51)["factor"]
    assert f["flops"] == pytest.approx(2 * 4096 ** 3 / 3)          # 4.58e10: the Cholesky and the inverse
    assert f["bound_ms_three_pass"] == pytest.approx(3 * f["bound_ms"], abs=2e-4)
    assert f["frac"] == pytest.approx(f["bound_ms"] / 1.51, abs=1e-4) and f["bar"] is None


def test_memory_bound_and_ragged_shapes():
    """Few rows: the bound is the bytes; a ragged last block and per-channel groups count."""
    r = bench.stage_rooflines(8, 4160, 1024, 3, -1, 128, syrk_ms=1.0, quantize_ms=1.0, peaks=PEAKS)
    q = r["column_loop_and_lazy_update"]
    nbytes = 2 * 8 * 4160 + 2 * 4160 * 4161 + 8 * 4160 * 3 / 8 + 8 * 8 * 1 + 4 * 4160
    assert q["bytes"] == int(nbytes)
    assert q["bound_ms"] == pytest.approx(nbytes / 6788.6e9 * 1e3, abs=1e-4)
    blocks = [(i, min(128, 4160 - i)) for i in range(0, 4160, 128)]
    assert blocks[-1] == (4096, 64)
    assert q["flops_lazy"] == sum(2 * 8 * nb * (4160 - i - nb) for i, nb in blocks)
    assert q["flops_in_block"] == sum(8 * nb * (nb - 1) for _, nb in blocks)
