"""CPU oracle (test infrastructure only): the plain definition of the routed MoE
expert layer with per-expert LoRA.  Imported by tests, the smoke check and the
benchmark's CPU-baseline leg; never by the product path."""
from .moe_lora_oracle import (  # noqa: F401
    RENORMALIZE, DEEPSEEK_V3, round_bf16, exp_f32, sigmoid_f32, route, align, silu,
    moe_lora_forward, pack_topk, unpack_topk, moe_lora_forward_routed,
    E4M3_MAX, FP8_BLOCK, e4m3_decode, round_e4m3, quant_act_fp8, dequant_act_fp8, fake_quant_act_fp8,
    dequant_weight_fp8, Fp8Experts, moe_lora_forward_fp8,
    E2M1_MAX, NVFP4_BLOCK, e2m1_decode, unpack_nvfp4, round_e2m1, quant_act_nvfp4, dequant_act_nvfp4,
    fake_quant_act_nvfp4, dequant_weight_nvfp4, Nvfp4Experts, moe_lora_forward_nvfp4,
)
