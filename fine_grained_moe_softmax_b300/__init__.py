"""B300 (sm_103a) DeepSeekMoE layer: forward, backward and the training pair.

The layer runs in hand-written CUDA kernels behind the C ABI of ``include/moe_b300.h``;
``binding`` exposes those entry points under their C names and ``layer.MoELayer`` holds the
device buffers (packed weights, workspace, outputs) for repeated calls.
"""
from .binding import (MOE_DTYPE_BF16, MOE_DTYPE_F32, N_STAGES, STAGE_NAMES, MoEConfig, MoEError,
                      moe_backward_workspace_bytes, moe_balance_stats, moe_combine,
                      moe_device_status, moe_expert_ffn, moe_launch_count, moe_layer_backward,
                      moe_layer_backward_saved, moe_layer_forward, moe_layer_forward_train,
                      moe_layer_routing,
                      moe_pack_weights, moe_pack_weights_backward, moe_packed_backward_bytes,
                      moe_packed_weight_bytes, moe_permute, moe_profile_enable, moe_profile_read,
                      moe_profile_read_gate_up,
                      moe_route, moe_selftest_bounded_wait, moe_status_string,
                      moe_workspace_bytes)
from .layer import MoELayer

__all__ = ["MOE_DTYPE_BF16", "MOE_DTYPE_F32", "N_STAGES", "STAGE_NAMES", "MoEConfig", "MoEError",
           "MoELayer", "moe_backward_workspace_bytes", "moe_balance_stats", "moe_combine",
           "moe_device_status", "moe_expert_ffn", "moe_launch_count", "moe_layer_backward",
           "moe_layer_backward_saved", "moe_layer_forward", "moe_layer_forward_train",
           "moe_layer_routing",
           "moe_pack_weights", "moe_pack_weights_backward", "moe_packed_backward_bytes",
           "moe_packed_weight_bytes", "moe_permute", "moe_profile_enable", "moe_profile_read",
           "moe_profile_read_gate_up",
           "moe_route", "moe_selftest_bounded_wait", "moe_status_string", "moe_workspace_bytes"]
