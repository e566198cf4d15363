"""GB300-native W4A16 routed mixture-of-experts layer.

The compute lives in libw4moe.so (hand-written CUDA for sm_103a, C ABI in
include/w4moe.h).  This package is its thin Python binding plus the seeded
synthetic workloads (``workloads``) used by the tests and the benchmark.

    import w4a16_moe_expert_sync_gb300 as w4
    q, s, z = w4.w4_quantize(W_fp32_cuda, group=128)
    ids, w = w4.w4_moe_route(logits, k=8)
    out = w4.w4_moe_layer(x_bf16, ids, w, (gu_q, gu_s, gu_z), (dn_q, dn_s, dn_z))
"""
from ._lib import (W4_DEV_BAD_EXPERT_ID, W4_DEV_FP16_RANGE, W4_DEV_OUT_OF_BOUNDS,
                   W4_DEV_PIPELINE_TIMEOUT,
                   W4_DEV_TOO_MANY_JOBS,
                   W4Error, header_functions, korder_to_natural, load_library,
                   w4_gather_activations, w4_grouped_gemm_down, w4_moe_align_gather,
                   w4_grouped_gemm_gate_up, w4_moe_align, w4_moe_align_capacity,
                   w4_moe_combine_fixed_order, w4_moe_combine_prepare,
                   w4_grouped_gemm_down_combine, w4_moe_layer, w4_moe_layer_static_scratch,
                   w4_moe_layer_workspace_size, w4_moe_layer_from_logits, w4_moe_layer_host,
                   w4_moe_layer_host_workspace_size,
                   w4_moe_route, w4_moe_route_align_gather, w4_quantize, w4_rmsnorm,
                   w4_sample_logits, w4_sample_logits_workspace_size, w4_fused_entropy,
                   w4_gumbel_argmax_sample, w4_w4a16_linear, w4_w4a16_linear_workspace_size)

__all__ = [
    "W4Error", "load_library", "header_functions", "korder_to_natural", "w4_gather_activations",
    "w4_moe_align_gather",
    "w4_quantize", "w4_moe_route", "w4_moe_align", "w4_moe_align_capacity",
    "w4_grouped_gemm_gate_up", "w4_grouped_gemm_down", "w4_moe_combine_fixed_order",
    "w4_moe_combine_prepare", "w4_grouped_gemm_down_combine",
    "w4_moe_layer", "w4_moe_layer_workspace_size", "w4_moe_layer_static_scratch",
    "w4_moe_layer_host", "w4_moe_layer_host_workspace_size",
    "w4_moe_route_align_gather", "w4_moe_layer_from_logits", "w4_rmsnorm", "w4_sample_logits",
    "w4_sample_logits_workspace_size", "w4_fused_entropy", "w4_gumbel_argmax_sample",
    "w4_w4a16_linear", "w4_w4a16_linear_workspace_size",
    "W4_DEV_BAD_EXPERT_ID", "W4_DEV_FP16_RANGE", "W4_DEV_OUT_OF_BOUNDS", "W4_DEV_PIPELINE_TIMEOUT", "W4_DEV_TOO_MANY_JOBS",
]
