"""CPU oracle for the Q4 MoE layer forward pass.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package; only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline / reference arm of ``bench.py`` use it.
"""
from .moe_oracle import (  # noqa: F401
    bf16_to_f64,
    unpack_codes,
    dequant,
    router_logits,
    select_experts,
    group_assignments,
    expert_ffn,
    hidden_sorted,
    moe_forward,
    silu,
)
