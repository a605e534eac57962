"""GB300 (sm_103a) row normalization: RMSNorm, fused residual add + RMSNorm,
LayerNorm and L2Norm on bf16 or fp16 rows, and fused Q/K RMSNorm + RoPE.

The compute lives in ``librownorm.so`` (CUDA kernels behind the C ABI of
``include/row_norm.h``); :mod:`row_normalization_gb300.binding` marshals torch
tensors into it.  Importing this package does not load the library; the first
call does, and fails loudly if it is not built.
"""
from .binding import (  # noqa: F401
    RN_DTYPE_BF16, RN_DTYPE_F16, RN_OP_ADD_RMSNORM, RN_OP_L2NORM, RN_OP_LAYERNORM, RN_OP_RMSNORM,
    RN_QK_AUTO, RN_QK_BULK, RN_ROPE_GPTJ, RN_ROPE_NEOX, RN_QK_FOUR_HEADS, RN_QK_HEAD_PER_WARP,
    RN_QK_PAIRS, RN_QK_PERSISTENT, RN_QK_TWO_HEADS,
    RN_SCHED_AUTO, RN_SCHED_CTA_ROW, RN_SCHED_PERSIST_BULK, RN_SCHED_WARP_ROW,
    RN_STATUS_BAD_POSITION, RN_STATUS_WAIT_TIMEOUT, RN_WORKSPACE_BYTES, RowNormError, add_rmsnorm_fwd,
    add_rmsnorm_select_schedule, device_status, error_string, l2norm_fwd, layernorm_fwd,
    layernorm_select_schedule, new_workspace, qk_norm_rope_fwd, qk_norm_rope_fwd_checked, qk_norm_rope_fwd_ex,
    qk_norm_rope_select_schedule, rmsnorm_fwd, rmsnorm_select_schedule, rope_cos_sin_table,
    row_norm_select_schedule, version)
