"""GB300-native fused Mixture-of-Experts expert layer with per-token
multi-LoRA adapters.

The compute path is libmlora.so (hand-written CUDA for sm_103a, C ABI in
include/mlora.h); this package holds its ctypes binding, the in-tree build
step and the seeded synthetic workload generator.
"""
from ._lib import (  # noqa: F401
    DEV_BAD_EXPERT_ID,
    DEV_BAD_LORA_IDX,
    DEV_BOUNDS,
    DEV_TIMEOUT,
    FORWARD_BLOCK_M,
    SCORE_SIGMOID_BIAS,
    SCORE_SOFTMAX,
    MloraError,
    declared_functions,
    load,
    mlora_moe_align,
    mlora_moe_align_max_padded,
    mlora_moe_forward,
    mlora_moe_forward_mxfp8,
    mlora_moe_forward_static,
    mlora_moe_read_status,
    mlora_moe_read_status_static,
    mlora_moe_route,
    mlora_moe_workspace_size,
    mlora_moe_workspace_size_mxfp8,
    mlora_mxfp8_quantize_weights,
    mlora_mxfp8_scales_size,
    mlora_set_stage_events,
    mlora_set_tile_config,
    mlora_set_pair_mode,
    mlora_pair_mode,
    mlora_tile_config,
    mlora_set_wait_test,
    mlora_status_string,
    STAGE_EVENTS,
    STAGE_NAMES,
)
