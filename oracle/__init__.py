"""CPU oracle (test infrastructure only): the plain definition of the routed MoE
expert layer with per-expert LoRA.  Imported by tests, the smoke check and the
benchmark's CPU-baseline leg; never by the product path."""
from .moe_lora_oracle import (  # noqa: F401
    RENORMALIZE, DEEPSEEK_V3, round_bf16, exp_f32, sigmoid_f32, route, align, silu,
    moe_lora_forward, pack_topk, unpack_topk, moe_lora_forward_routed,
)
