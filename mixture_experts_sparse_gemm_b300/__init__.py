"""Single-GPU sparsely-gated Mixture-of-Experts SwiGLU FFN forward for NVIDIA B300.

The compute lives in ``libmoe_b300.so`` (hand-written CUDA for sm_103a, C ABI in
``include/moe_b300.h``).  ``binding`` marshals torch tensors into those entry
points; ``layer`` allocates the buffers a layer needs around them.
"""
from .binding import (EXPORTS, MoeError, config, config_from_workload, lib, moe_buffer_rows,  # noqa: F401
                      moe_check_device_error, moe_combine, moe_config, moe_dispatch, moe_expert_capacity,
                      moe_forward, moe_grouped_ffn, moe_grouped_ffn_down, moe_grouped_ffn_up,
                      moe_launch_count, moe_load_stats, moe_pack_weights, moe_packed_weights_size, moe_route,
                      moe_validate_config, moe_workspace_size, status_string)
