"""GB300-native memory-bound training-step kernels.

``libtb.so`` (built from ``csrc/`` for sm_103a) implements the fused
mixed-precision multi-tensor AdamW step, the row-wise softmax backward and the
LayerNorm backward behind the C ABI declared in ``include/tb.h``.  This package
is its thin Python binding (same names as the C entry points) plus the seeded
synthetic-input module ``synth``.
"""
from ._binding import (  # noqa: F401
    EXPORTS, STATUS, TB_BF16, TB_F16, TB_F32, AdamWPlan, TbError, library_path,
    tb_adamw_grad_norm, tb_adamw_grad_norm_workspace_size, tb_adamw_plan_create,
    tb_adamw_plan_destroy, tb_adamw_selftest_stale_counter, tb_adamw_step, tb_adamw_step_clipped,
    tb_adamw_step_device,
    tb_cast_from_f32, tb_cast_to_f32,
    tb_device_error,
    tb_layernorm_bwd, tb_layernorm_bwd_noalloc, tb_layernorm_bwd_selftest_timeout,
    tb_layernorm_bwd_workspace_size,
    tb_rmsnorm_bwd, tb_rmsnorm_bwd_workspace_size, tb_softmax_bwd, tb_softmax_bwd_causal,
    tb_status_string, tb_version,
)
