"""ZeRO partitioned mixed-precision optimizer step for NVIDIA GB300 (sm_103a).

The data-parallel hot path of ZeRO: the model states are flattened into one
padded buffer and partitioned over Nd ranks, and one rank's shard is updated
by hand-written CUDA kernels (gradient accumulation; unscale + overflow +
global squared norm; clip + AdamW + cast to fp16/bf16).  Around the step:
the stage-2 gradient reduction fused with the norm pass, the stage-3
parameter gather (shards back to tensors) with its per-layer plan, the
offload step on the host cores, and 1-bit Adam's compression stage.  The C ABI is in
``include/zero_pml.h``; this package is its Python binding.
"""
from .binding import (  # noqa: F401
    HParams,
    Layout,
    ZeroError,
    ZERO_ECAPTURE,
    ZERO_BF16,
    ZERO_F16,
    ZERO_F32,
    STATE_BYTES,
    TensorList,
    LIB_PATH,
    lib,
    new_state,
    new_workspace,
    parse_state,
    OffloadScalars,
    default_host_threads,
    zero_accumulate_grads,
    zero_accumulate_grads_norm,
    zero_offload_apply,
    zero_offload_copy,
    zero_offload_decide,
    zero_adam_step,
    zero_grad_norm_overflow,
    zero_partition_layout,
    zero_state_init,
    zero_reduce_grads,
    zero_step,
    ListPlan,
    zero_list_prepare,
    zero_step_prepared,
    zero_strerror,
    zero_workspace_bytes,
    zero_workspace_stalls,
    GatherPlan,
    zero_gather_params,
    zero_gather_plan,
    zero_gather_workspace_bytes,
    zero_scatter_params,
    zero_onebit_server,
    zero_onebit_update,
    zero_onebit_worker,
)
