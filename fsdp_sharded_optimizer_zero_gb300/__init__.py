"""GB300-native data-parallel optimizer step (DDP / ZeRO-1/2/3 / FSDP) on one GPU.

The N data-parallel ranks are simulated as separate device buffers. The work is done by
hand-written sm_103a CUDA kernels behind a C ABI (include/zero.h, libzero_gb300.so); this
package is the thin Python binding with the same entry-point names.
"""
from ._lib import (  # noqa: F401
    EXPORTS, LIB_PATH, STAGE_IDS, ZERO_ALL_RANKS, ZERO_MAX_RANKS, ZERO_RANK_VIEW, Plan, ZeroError,
    FSDP_BACKWARD_PREFETCH, FSDP_GATHER_MATERIALIZE, FSDP_OVERLAP_OPTIMIZER, FSDP_SEPARATE_OPTIMIZER, ddp_allreduce, fsdp_gather_rows, fsdp_mlp_forward, fsdp_transpose_cat, fsdp_unit_backward, fsdp_unit_backward_workspace, fsdp_unit_forward, fsdp_unit_forward_static_scratch, fsdp_zero3_mlp_step, fsdp_zero3_mlp_step_workspace, fsdp_zero3_step, fsdp_zero3_step_workspace, library, zero_adam_step, zero_allgather_params,
    zero_bucket_range, zero_device_status, zero_fused_step, zero_fused_step_buckets, zero_fused_step_fp32_grads, zero_fused_step_host, zero_last_error,
    zero_plan, zero_plan_check_memory, zero_plan_query, zero_reduce_scatter, zero_selftest_bounded_wait, zero_set_fused_kernel, zero_set_gemm_kernel, zero_version,
)
