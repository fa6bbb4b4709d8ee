"""GB300-native sharded optimizer step (ZeRO-1/2/3 update) on one GPU.

The N data-parallel ranks are N resident HBM buffers; the reduce-scatter, the
per-rank AdamW on fp32 master/m/v shards, the bf16 cast and the all-gather run
in hand-written sm_103a kernels behind a C ABI (include/zero.h).  This package
is its thin Python binding.  The library is loaded on first use and must have
been built (build.build()); there is no CPU fallback.
"""
from .binding import (AdamW, OffloadEngine, UnitSteps, ZeroError, ZeroPlan, ZERO_BF16, ZERO_F32, ZERO_MAX_RANKS, lib, rank_buffers, zero_adamw_shard_step,
                      zero_adamw_shard_step_clipped, zero_all_gather, zero_all_gather_bf16, zero_all_gather_unit, zero_bias_corrections, zero_clip_finalize, zero_clip_reduce_unit, zero_clip_reduce_units, zero_grad_sqnorm,
                      zero_offload_adamw, zero_offload_create, zero_offload_destroy, zero_offload_info, zero_offload_step,
                      zero_offload_timings, zero_plan_attach,
                      zero_plan_align, zero_plan_counts, zero_plan_create, zero_plan_create_aligned, zero_plan_check, zero_plan_destroy, zero_plan_device_errors, zero_plan_query, zero_plan_segments, zero_plan_local_segments,
                      zero_plan_workspace_bytes, zero_reduce_scatter, zero_reduce_scatter_unit, zero_reshard, zero_step, zero_step_unit, zero_step_units)

__all__ = ["AdamW", "OffloadEngine", "UnitSteps", "ZeroError", "ZeroPlan", "ZERO_BF16", "ZERO_F32", "ZERO_MAX_RANKS", "lib", "rank_buffers",
           "zero_adamw_shard_step", "zero_adamw_shard_step_clipped", "zero_all_gather", "zero_all_gather_bf16", "zero_all_gather_unit", "zero_bias_corrections", "zero_clip_finalize", "zero_clip_reduce_unit", "zero_clip_reduce_units",
           "zero_grad_sqnorm", "zero_offload_adamw", "zero_offload_create", "zero_offload_destroy", "zero_offload_info",
           "zero_offload_step", "zero_offload_timings", "zero_plan_align", "zero_plan_attach", "zero_plan_counts", "zero_plan_create", "zero_plan_create_aligned", "zero_plan_check", "zero_plan_destroy", "zero_plan_device_errors",
           "zero_plan_query", "zero_plan_segments", "zero_plan_local_segments", "zero_plan_workspace_bytes", "zero_reduce_scatter", "zero_reduce_scatter_unit", "zero_reshard", "zero_step", "zero_step_unit", "zero_step_units"]
