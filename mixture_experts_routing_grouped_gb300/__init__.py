"""GB300-native (sm_103a) fused, grouped-routed MoE layer forward.

The computation lives in hand-written CUDA kernels behind the C ABI of
include/moe_gb300.h (libmoe_gb300.so, built in-tree by ``build.build()``). This
package is the thin Python binding: torch tensors in, raw pointers and the
current CUDA stream out. There is no CPU or PyTorch fallback: if the library is
missing, every call raises.
"""
from ._binding import (  # noqa: F401
    DEVERR_EXPERT_ID, DEVERR_GROUP_META, DEVERR_TIMEOUT, MoeError, exported_symbols, gmm_lowp,
    gmm_lowp_workspace_size, lib,
    moe_align_block_size, moe_align_max_padded, moe_check_device_error, moe_fused_forward,
    moe_fused_forward_fp8, moe_fused_forward_fp8_workspace_size,
    moe_fused_forward_noalloc, moe_fused_forward_noalloc_check_error, moe_fused_forward_workspace_size, moe_grouped_topk, moe_quant_per_token, moe_read_probe, moe_router_topk,
    moe_router_topk_workspace_size, moe_set_stage_events, moe_wait_timeout_probe,
    status_string,
)
