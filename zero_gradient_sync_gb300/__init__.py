"""GB300-native fused data-parallel step: gradient accumulation, ring-order reduce-scatter, averaging with
loss-scale unscaling and a global non-finite skip, ZeRO-partitioned mixed-precision Adam, and the bf16
parameter all-gather -- all n replicas' buffers in one GPU's memory.

The computation lives in libdpstep.so (CUDA, sm_103a; C ABI in include/dpstep.h).  This package is its
binding; importing it without the built library raises ImportError.
"""
from ._lib import (  # noqa: F401
    DP_ERR_ALIGNMENT, DP_ERR_CUDA, DP_ERR_INVALID_ARG, DP_ERR_IO, DP_ERR_TIMEOUT, DP_MAX_N, DP_MAX_NA, DP_MAX_SEG,
    DP_DEFER_COMMIT, DP_DEVICE_SCALE, DP_KERNEL_SEG, DP_OK, DP_ORDER_RING, DP_ORDER_TREE, DP_SUM_COMPENSATED, DP_SUM_PLAIN, LIB, LIB_PATH, STATE_BYTES, DPError,
    Layout, adam, dp_accumulate, dp_adam_shard, dp_allgather_params, dp_checkpoint_info, dp_checkpoint_load,
    dp_checkpoint_save, dp_commit_single_pass, dp_commit_step, dp_get_wait_timeout_ns, dp_global_batch, dp_kernel_launches, dp_memory_model,
    dp_read_status, dp_reduce_scatter_avg, dp_reduce_scatter_micro, dp_scaler_init, dp_selftest_wait_timeout, dp_set_wait_timeout_ns,
    dp_state_init, dp_step, dp_step_from_host, dp_step_reduce, dp_step_scaled, dp_step_single_pass,
    dp_step_single_pass_from_host, dp_step_static, dp_step_update,
    dp_traffic_model, new_state, read_state, scaler)
