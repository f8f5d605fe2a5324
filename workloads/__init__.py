"""Seeded synthetic workloads for the MoE layer.

This package is shared by the CPU oracle harness and the GPU harness. It holds the
random draws and the rounding of those draws to their storage types, and nothing of
the layer's own arithmetic.
"""
from .configs import CONFIGS, LayerConfig, get_config  # noqa: F401
from .synth import (  # noqa: F401
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_dy,
    make_logits,
    make_w13,
    make_w2,
    make_x,
    normal_f32,
    normal_f32_rows,
)
