"""GB300 (sm_103a) selective log-prob + GRPO loss forward/backward library.

Python face of the C ABI declared in ``include/grpo_gb300.h``; all compute
runs in the CUDA library ``libgrpo_gb300.so`` built from ``csrc/``.
"""

from ._binding import (  # noqa: F401
    EXPORTED,
    GRPO_ERR_BAD_TOKEN_ID,
    GRPO_ERR_DEVICE_TIMEOUT,
    GRPO_ERR_NONFINITE,
    GRPO_OK,
    NOALLOC_MAX_TOKENS,
    GrpoError,
    GrpoParams,
    GrpoShape,
    alloc_workspace,
    grpo_get_plan,
    grpo_launch_timing_enable,
    grpo_launch_timing_read,
    grpo_logp_fwd,
    grpo_logp_fwd_noalloc,
    grpo_loss_fwd_bwd,
    grpo_read_device_status,
    grpo_selftest_bounded_wait,
    grpo_workspace_size,
    lib,
    make_params,
    make_shape,
    status_string,
)
