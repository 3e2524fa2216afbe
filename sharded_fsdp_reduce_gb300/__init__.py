"""GB300-native FSDP FlatParameter step: flatten/pad, fused reduce-scatter +
AdamW + cast, all-gather and unflatten, as hand-written sm_103a CUDA behind a
C ABI (include/fsdp.h). This package is the thin Python binding over it.
"""
from .fsdp import (OPTIMIZERS, AdamWHParams, FsdpError, StepConfig, StepGraph, StepPlan, UnitDescs, View, dtype_code,
                   fsdp_all_gather, fsdp_check_bounded_wait, fsdp_flatten_pad, fsdp_last_cuda_error,
                   fsdp_padded_numel, fsdp_reduce_scatter_adam_cast, fsdp_reduce_scatter_adam_cast_gather,
                   fsdp_reduce_scatter_step, fsdp_status_string, fsdp_step_units, fsdp_step_units_ex,
                   fsdp_step_units_ex_launches, fsdp_step_units_launches, fsdp_take_wait_timeouts,
                   fsdp_unflatten_views)
from .unit import FlatParamUnit, UnitSequence

__all__ = [
    "AdamWHParams", "StepConfig", "OPTIMIZERS", "FsdpError", "View", "FlatParamUnit", "UnitSequence", "dtype_code",
    "fsdp_padded_numel", "fsdp_unflatten_views", "fsdp_flatten_pad", "fsdp_reduce_scatter_adam_cast",
    "fsdp_reduce_scatter_adam_cast_gather", "fsdp_reduce_scatter_step", "fsdp_all_gather",
    "fsdp_status_string", "fsdp_last_cuda_error", "fsdp_take_wait_timeouts", "fsdp_check_bounded_wait",
    "UnitDescs", "fsdp_step_units", "fsdp_step_units_ex", "StepGraph", "StepPlan", "fsdp_step_units_launches",
    "fsdp_step_units_ex_launches",
]
