"""GB300-native ZeRO-1/2 mixed-precision AdamW step.

R data-parallel ranks are emulated as R buffers in one GPU's HBM; one call
reduce-scatters their bf16 gradients in fixed rank order with fp32
accumulation, updates each rank's shard of the fp32 master weights and Adam
moments, and all-gathers the bf16 result into every rank's replica.  The
work runs in the hand-written sm_103a kernels of libzero_step.so (C ABI in
include/zero_step.h); this package is its thin binding.
"""
from .binding import (  # noqa: F401
    EXPORTED, Plan, ZeroError, hparams, lib, zero_abi_version, zero_adamw_shard, zero_ag_cast,
    zero_plan_create, zero_plan_destroy, zero_plan_owner, zero_rs_avg, zero_status_string,
    zero_step, zero_step_host, zero_step_staged_noalloc, zero_step_clipped,
    zero_clip_scratch_bytes, ZERO_DEV_SKIPPED, ZERO_FLAG_SKIP_NONFINITE, zero3_step, zero3_gather,
    zero_ckpt_write_host, zero_ckpt_read_host, zero_ckpt_save_async, zero_ckpt_job_wait,
    zero_ckpt_load, zero_step_compressed, zero_check_replicas, zero_step_onebit, zero3_rs_unit, zero3_update, zero_get_device_status, zero3_gather_units,
    gather_unit_table, ZERO_MAX_GATHER_UNITS,
    ZERO_DEV_DRAIN_FAILED, ZERO_COMP_FP16, ZERO_COMP_INT8, ZERO_COMP_SIGN, ZERO_DEV_NONFINITE, ZERO_FLAG_CHECK_FINITE, ZERO_VARIANT_FUSED,
    ZERO_VARIANT_STAGED, ZERO_VARIANT_FUSED_TMA, ZERO_DEV_TIMEOUT, ZERO_FLAG_DEBUG_EXPIRE_WAITS,
)
