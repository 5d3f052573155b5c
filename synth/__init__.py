"""Seeded synthetic inputs (layer weights and calibration activations).

This package only draws inputs. It holds none of GPTQ's arithmetic, so the CPU
oracle and the CUDA path can both consume the exact bytes it produces.
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    LayerSpec,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_weight,
    make_activations,
    gen_activations_into,
    workload,
    small_layer,
    ActSpec,
)
