"""Seeded synthetic inputs for the Q4 MoE layer (shared by the tests, the bench and the oracle checks).

This package only draws random numbers and stores them in the canonical formats; it holds none
of the layer's arithmetic.
"""
from .moe_inputs import (  # noqa: F401
    LayerShape,
    FULL,
    TINY,
    STACK_LAYERS,
    STACK_DECODE_STEPS,
    CONFIGS,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_layer,
    make_tokens,
    zipf_router_bias,
)
