"""Seeded synthetic layers and token batches in the canonical (MLX-style affine Q4) format.

Everything here is a random draw or a storage conversion; nothing computes the MoE layer.

Canonical formats (the checkpoint format the pages name: "MLX affine 4-bit, group size 64",
agentnative.dev, section "Setup"; "every group of 64 weights shares a bfloat16 scale and bias",
section "Prefill: keep routing on the GPU, dequantize in flight"):

* bf16 values are carried as ``uint16`` bit patterns.
* A quantized matrix ``W[rows, cols]`` (``cols`` = input dimension) is the triple
  ``q uint32[rows, cols/8]`` (code of column ``c`` in bits ``4*(c%8)`` of word ``c//8``,
  i.e. low nibble first along the input dimension), ``scale uint16[rows, cols/64]`` and
  ``bias uint16[rows, cols/64]``.
* Routed experts are stacked along a leading expert axis; the shared expert has none.

Input recipe (the synthetic workloads of the layer shape d=2048, 256 experts, top-8, I=512):
x ~ N(0,1); router weight ~ N(0, 1/d); codes uniform in 0..15; scale ~ U(0.01, 0.03);
bias = -8*scale; all rounded to bf16 with round-to-nearest-even. The skewed workload adds a
per-expert router bias 2*ln(p_r), p_r the Zipf(s=1.1) probability of rank r = e+1.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Tags that separate the random streams of the different tensors of one seed.
_TAG_X = 1
_TAG_ROUTER = 2
_TAG_Q = {"gate": 10, "up": 11, "down": 12, "sh_gate": 13, "sh_up": 14, "sh_down": 15}
_TAG_S = {k: v + 10 for k, v in _TAG_Q.items()}


@dataclasses.dataclass(frozen=True)
class LayerShape:
    d: int = 2048          # hidden size
    n_experts: int = 256   # routed experts E
    top_k: int = 8         # experts picked per token
    inter: int = 512       # routed-expert intermediate size I
    shared_inter: int = 512  # shared-expert intermediate size
    group: int = 64        # quantization group along the input dimension


TINY = LayerShape(d=256, n_experts=16, top_k=2, inter=128, shared_inter=128)
FULL = LayerShape()

# name -> (shape, tokens, router bias kind)
CONFIGS = {
    "tiny": (TINY, 4, None),
    "decode": (FULL, 1, None),
    "prefill512": (FULL, 512, None),
    "skew2048": (FULL, 2048, "zipf"),
    "stack_prefill": (FULL, 4096, None),
}
STACK_LAYERS = 40
STACK_DECODE_STEPS = 256


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(entropy=seed, spawn_key=(tag,))))


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def zipf_router_bias(n_experts: int, s: float = 1.1, strength: float = 2.0) -> np.ndarray:
    """Per-expert router bias strength*ln(p_r) with p_r the Zipf(s) probability of rank r=e+1."""
    ranks = np.arange(1, n_experts + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    return (strength * np.log(p)).astype(np.float32)


def _q4_matrix(seed: int, name: str, lead: tuple, rows: int, cols: int, group: int):
    """Random codes (uniform 0..15), scale ~ U(0.01,0.03) and bias = -8*scale, canonical layout."""
    words = _rng(seed, _TAG_Q[name]).integers(0, 2**32, size=lead + (rows, cols // 8),
                                              dtype=np.uint32, endpoint=False)
    scale_f = _rng(seed, _TAG_S[name]).uniform(0.01, 0.03, size=lead + (rows, cols // group))
    scale = f32_to_bf16_bits(scale_f.astype(np.float32))
    bias = f32_to_bf16_bits(np.float32(-8.0) * bf16_bits_to_f32(scale))  # exact in bf16
    return {"q": words, "scale": scale, "bias": bias}


def make_layer(shape: LayerShape, seed: int = 0, router_bias: str | None = None) -> dict:
    """One MoE layer's parameters in the canonical format (numpy, host memory)."""
    d, E, I, Is, g = shape.d, shape.n_experts, shape.inter, shape.shared_inter, shape.group
    wr = _rng(seed, _TAG_ROUTER).standard_normal((E, d), dtype=np.float32) * np.float32(1.0 / math.sqrt(d))
    layer = {
        "shape": shape,
        "router_w": f32_to_bf16_bits(wr),
        "router_bias": zipf_router_bias(E) if router_bias == "zipf" else None,
        "gate": _q4_matrix(seed, "gate", (E,), I, d, g),
        "up": _q4_matrix(seed, "up", (E,), I, d, g),
        "down": _q4_matrix(seed, "down", (E,), d, I, g),
        "sh_gate": _q4_matrix(seed, "sh_gate", (), Is, d, g),
        "sh_up": _q4_matrix(seed, "sh_up", (), Is, d, g),
        "sh_down": _q4_matrix(seed, "sh_down", (), d, Is, g),
    }
    if router_bias not in (None, "zipf"):
        raise ValueError(f"unknown router bias kind {router_bias!r}")
    return layer


def make_tokens(n_tokens: int, d: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Hidden states x ~ N(0,1) rounded to bf16, as uint16 bits [n_tokens, d]."""
    x = _rng(seed * 1_000_003 + stream, _TAG_X).standard_normal((n_tokens, d), dtype=np.float32)
    return f32_to_bf16_bits(x)
