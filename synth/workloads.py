"""Seeded synthetic layers and calibration activations for the GPTQ per-layer path.

The pages calibrate on 128 web-text sequences of 2048 tokens ("GPTQ: fixing errors
as you go", example "a 4-bit Llama layer"; "GPTQ-style round-to-nearest with Hessian
weighting", section "Computing the Hessian") and quantize Llama/OPT/BLOOM layers. No
dataset or trained weight is available, so every input here is drawn from seeded
generators with the same shapes and with heavy-tailed, correlated, outlier-channel
statistics. Nothing in this file computes any part of GPTQ.

Reproducibility: every draw comes from numpy's PCG64 seeded by a
``SeedSequence(seed, spawn_key=(tag, index))``. Activations are generated in chunks
of ``CHUNK`` tokens, each chunk from its own key, so a chunk can be regenerated on
its own and chunks can be drawn in parallel threads with identical results on the
x86 and the Arm host.

All values are produced in float32 and rounded once to bfloat16 (round to nearest,
ties to even); both the oracle and the CUDA path consume those bf16 bytes.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK = 4096          # tokens per independently seeded activation chunk
ROW_CHUNK = 1024      # weight rows per independently seeded chunk

# spawn-key tags
_TAG_PARAMS = 0
_TAG_X = 1
_TAG_W = 2


# ----------------------------------------------------------------------------------
# bfloat16 bytes
# ----------------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits (uint16) to the float32 values they encode (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, tag: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(tag, index)))


def _threads(threads: int | None) -> int:
    if threads is not None:
        return max(1, int(threads))
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------------
# weights
# ----------------------------------------------------------------------------------
def make_weight(m: int, d: int, seed: int, layer: int = 0, std: float = 0.02,
                threads: int | None = None) -> np.ndarray:
    """W (m x d, out x in) with iid N(0, std^2) entries, as bf16 bits (uint16)."""
    out = np.empty((m, d), dtype=np.uint16)
    nchunks = (m + ROW_CHUNK - 1) // ROW_CHUNK

    def one(c: int) -> None:
        r0, r1 = c * ROW_CHUNK, min(m, (c + 1) * ROW_CHUNK)
        rng = _rng(seed, _TAG_W, layer * 1_000_003 + c)
        w = rng.standard_normal((r1 - r0, d), dtype=np.float32) * np.float32(std)
        out[r0:r1] = f32_to_bf16_bits(w)

    with ThreadPoolExecutor(_threads(threads)) as ex:
        list(ex.map(one, range(nchunks)))
    return out


# ----------------------------------------------------------------------------------
# activations
# ----------------------------------------------------------------------------------
@dataclass(frozen=True)
class ActSpec:
    """Recipe of one calibration-activation stream (one Hessian)."""
    kind: str            # "gauss_cov" | "heavy_tail" | "silu_gate"
    n: int               # tokens
    d: int               # input channels
    seed: int
    stream: int = 0      # distinguishes Hessians of one workload
    outlier_frac: float = 0.01
    outlier_count: int | None = None   # overrides outlier_frac when given
    outlier_scale: float = 30.0
    rank: int = 64


def _student_t4_unit(rng: np.random.Generator, shape) -> np.ndarray:
    """Student-t with 4 degrees of freedom scaled to unit variance (t_4 / sqrt 2).

    t_4 = Z / sqrt(V/4) with V ~ chi^2_4 = 2 Gamma(2, 1); dividing by sqrt(2) gives
    Z / sqrt(G) with G ~ Gamma(2, 1).
    """
    z = rng.standard_normal(shape, dtype=np.float32)
    g = rng.standard_gamma(2.0, shape, dtype=np.float32)
    return z / np.sqrt(g)


def _params(spec: ActSpec):
    rng = _rng(spec.seed, _TAG_PARAMS, spec.stream)
    d = spec.d
    n_out = spec.outlier_count if spec.outlier_count is not None else int(round(spec.outlier_frac * d))
    if spec.kind == "gauss_cov":
        a = rng.standard_normal((d, d))
        sigma = a @ a.T / d + 0.1 * np.eye(d)
        chol = np.linalg.cholesky(sigma).astype(np.float32)
        mix = (chol,)
    elif spec.kind == "heavy_tail":
        mix = (rng.standard_normal((spec.rank, d), dtype=np.float32),)
    elif spec.kind == "silu_gate":
        mix = (rng.standard_normal((spec.rank, d), dtype=np.float32),
               rng.standard_normal((spec.rank, d), dtype=np.float32))
    else:
        raise ValueError(f"unknown activation kind {spec.kind!r}")
    outliers = np.sort(rng.choice(d, size=n_out, replace=False)) if n_out > 0 else np.zeros(0, np.int64)
    return mix, outliers


def _chunk_f32(spec: ActSpec, mix, outliers, c: int) -> np.ndarray:
    t0, t1 = c * CHUNK, min(spec.n, (c + 1) * CHUNK)
    rows = t1 - t0
    rng = _rng(spec.seed, _TAG_X, spec.stream * 1_000_003 + c)
    inv_sqrt_r = np.float32(1.0 / np.sqrt(spec.rank))
    if spec.kind == "gauss_cov":
        (chol,) = mix
        z = rng.standard_normal((rows, spec.d), dtype=np.float32)
        x = z @ chol.T
    elif spec.kind == "heavy_tail":
        (m,) = mix
        tz = _student_t4_unit(rng, (rows, spec.rank))
        te = _student_t4_unit(rng, (rows, spec.d))
        x = (tz @ m) * inv_sqrt_r + np.float32(0.5) * te
    else:  # silu_gate: SiLU(g) * u with Gaussian low-rank + noise g and u
        mg, mu = mix
        g = (rng.standard_normal((rows, spec.rank), dtype=np.float32) @ mg) * inv_sqrt_r \
            + np.float32(0.5) * rng.standard_normal((rows, spec.d), dtype=np.float32)
        u = (rng.standard_normal((rows, spec.rank), dtype=np.float32) @ mu) * inv_sqrt_r \
            + np.float32(0.5) * rng.standard_normal((rows, spec.d), dtype=np.float32)
        x = g / (np.float32(1.0) + np.exp(-g)) * u
    if outliers.size:
        x[:, outliers] *= np.float32(spec.outlier_scale)
    return x.astype(np.float32, copy=False)


def gen_activations_into(spec: ActSpec, out: np.ndarray, threads: int | None = None,
                         token_range: tuple[int, int] | None = None) -> np.ndarray:
    """Write bf16 bits of X (spec.n x spec.d, token-major) into ``out``.

    ``token_range`` restricts generation to whole chunks ``[t0, t1)`` (both multiples
    of CHUNK, or t1 == n); ``out`` then holds only those rows.
    """
    t0, t1 = (0, spec.n) if token_range is None else token_range
    if t0 % CHUNK or (t1 % CHUNK and t1 != spec.n):
        raise ValueError("token_range must be chunk aligned")
    if out.shape != (t1 - t0, spec.d) or out.dtype != np.uint16:
        raise ValueError(f"out must be uint16 of shape {(t1 - t0, spec.d)}")
    mix, outliers = _params(spec)
    c0, c1 = t0 // CHUNK, (t1 + CHUNK - 1) // CHUNK

    def one(c: int) -> None:
        x = _chunk_f32(spec, mix, outliers, c)
        r0 = c * CHUNK - t0
        out[r0:r0 + x.shape[0]] = f32_to_bf16_bits(x)

    with ThreadPoolExecutor(_threads(threads)) as ex:
        list(ex.map(one, range(c0, c1)))
    return out


def make_activations(spec: ActSpec, threads: int | None = None) -> np.ndarray:
    """X (n x d, token-major) as bf16 bits (uint16)."""
    out = np.empty((spec.n, spec.d), dtype=np.uint16)
    return gen_activations_into(spec, out, threads)


# ----------------------------------------------------------------------------------
# named workloads
# ----------------------------------------------------------------------------------
@dataclass(frozen=True)
class LayerSpec:
    name: str
    m: int          # output features (rows of W)
    d: int          # input features (columns of W)
    hessian: str    # key into Workload.acts: layers that see the same inputs share H
    index: int      # weight seed index


@dataclass(frozen=True)
class Workload:
    name: str
    layers: tuple
    acts: dict = field(default_factory=dict)
    bits: int = 4
    group_size: int = 128          # -1: one scale/zero per output row
    blocksize: int = 128
    percdamp: float = 0.01
    act_order: bool = False
    seed: int = 0
    description: str = ""

    def weight(self, layer: LayerSpec, threads: int | None = None) -> np.ndarray:
        return make_weight(layer.m, layer.d, self.seed, layer.index, threads=threads)


def _c0() -> Workload:
    acts = {"in": ActSpec("gauss_cov", 512, 256, seed=0, outlier_count=4, outlier_scale=20.0)}
    return Workload("toy_256", (LayerSpec("linear", 256, 256, "in", 0),), acts,
                    bits=4, group_size=128, seed=0,
                    description="256x256 layer, 512 Gaussian correlated tokens, 4 outlier channels x20")


def _c1(seed: int = 1) -> dict:
    return {"in": ActSpec("heavy_tail", 262144, 4096, seed=seed)}


WORKLOADS = {
    "toy_256": _c0(),
    "llama_4096_g128": Workload(
        "llama_4096_g128", (LayerSpec("proj", 4096, 4096, "in", 0),), _c1(), bits=4,
        group_size=128, seed=1,
        description="Llama-style 4096x4096 projection, 262144 heavy-tailed tokens, 4-bit g128"),
    "llama_4096_3bit_actorder": Workload(
        "llama_4096_3bit_actorder", (LayerSpec("proj", 4096, 4096, "in", 0),), _c1(), bits=3,
        group_size=-1, act_order=True, seed=1,
        description="same layer and tokens, 3-bit per-channel with act-order"),
    "llama7b_mlp": Workload(
        "llama7b_mlp",
        (LayerSpec("gate", 11008, 4096, "mlp_in", 0), LayerSpec("up", 11008, 4096, "mlp_in", 1),
         LayerSpec("down", 4096, 11008, "mlp_down", 2)),
        {"mlp_in": ActSpec("heavy_tail", 262144, 4096, seed=3, stream=0),
         "mlp_down": ActSpec("silu_gate", 262144, 11008, seed=3, stream=1)},
        bits=4, group_size=128, seed=3, description="Llama-7B MLP, 4-bit g128"),
    "llama70b_block": Workload(
        "llama70b_block",
        (LayerSpec("q", 8192, 8192, "attn_in", 0), LayerSpec("k", 1024, 8192, "attn_in", 1),
         LayerSpec("v", 1024, 8192, "attn_in", 2), LayerSpec("o", 8192, 8192, "attn_out", 3),
         LayerSpec("gate", 28672, 8192, "mlp_in", 4), LayerSpec("up", 28672, 8192, "mlp_in", 5),
         LayerSpec("down", 8192, 28672, "mlp_down", 6)),
        {"attn_in": ActSpec("heavy_tail", 131072, 8192, seed=4, stream=0),
         "attn_out": ActSpec("heavy_tail", 131072, 8192, seed=4, stream=1),
         "mlp_in": ActSpec("heavy_tail", 131072, 8192, seed=4, stream=2),
         "mlp_down": ActSpec("silu_gate", 131072, 28672, seed=4, stream=3)},
        bits=4, group_size=128, seed=4, description="70B-shaped decoder block, 4-bit g128 (2-bit g64 variant)"),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def small_layer(m: int, d: int, n: int, seed: int, kind: str = "heavy_tail",
                outlier_count: int | None = None):
    """A reduced-size layer from the same recipes, for parity tests: (W bits, X bits)."""
    spec = ActSpec(kind, n, d, seed=seed, outlier_count=outlier_count)
    return make_weight(m, d, seed, 0), make_activations(spec)
