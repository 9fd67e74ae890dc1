"""Routed MoE expert layer with per-expert LoRA for GB300 (sm_103a).

The compute path is the CUDA library libmoelora.so (C ABI in include/moe_lora.h);
`binding` marshals torch tensors into it.  `workloads` draws seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    Handle, MoELoRAError, alloc_workspace, lib, make_args, moe_lora_check_status, moe_lora_create,
    moe_lora_forward, moe_lora_forward_fp8, moe_lora_forward_routed, moe_lora_grouped_gemm_fp8, moe_lora_permute,
    moe_lora_quant_fp8, moe_lora_route, moe_lora_forward_nvfp4, moe_lora_quant_nvfp4, moe_lora_grouped_gemm_nvfp4,
    moe_lora_status_string, moe_lora_validate, moe_lora_pack_lora_b, moe_lora_packed_lora_b_size,
    packed_lora_b_shape, moe_lora_pack_lora_a, moe_lora_packed_lora_a_size, packed_lora_a_shape,
    moe_lora_workspace_size, FLAG_LORA_OFF, FLAG_FORCE_SINGLE_STREAM, FLAG_FORCE_TWO_STREAM, FLAG_UNFUSED_LORA, FLAG_NO_PDL, FLAG_SHARED_OUTER,
    FLAG_DOWN_LORA_SIDE, FLAG_SEPARATE_SHRINK,
    ROUTE_RENORMALIZE, ROUTE_DEEPSEEK_V3, STAGES, NUM_STAGES,
)
