"""GB300-native (sm_103a) ZeRO / FSDP sharded mixed-precision step over a
FlatParameter, with all N_d logical data-parallel ranks held in one GPU.

The compute lives in the CUDA library declared by ``include/zero_flat.h``;
``zero`` is its thin ctypes binding (same function names), ``buffers`` lays
out per-rank device buffers with PyTorch allocations, ``synthetic`` draws the
seeded synthetic workloads, and ``build`` compiles the library in-tree.
"""
from .zero import (ZERO_MAX_RANKS, zero1_accumulate, zero1_step, zero_param_layout,
                   zero_shard_numel, ZeroAdamW, ZeroError, ZeroLayout, load, zero_abi_version,
                   zero_adamw_shard_step, zero_all_gather, zero_device_status, zero_flat_layout,
                   zero_flatten, zero_last_error, zero_reduce_scatter, zero_selftest_wait_timeout,
                   zero_shard_segments, zero_step, zero_step_units, zero_step_units_clip,
                   zero_step_units_clip_noalloc, zero_clip_workspace_bytes, zero_unflatten,
                   zero_step_units_host, HostTables, ZERO_HOST_GRADS_FREE,
                   ZERO_HOST_SM_COPY)

__all__ = [
    "ZERO_MAX_RANKS", "zero1_accumulate", "zero1_step", "zero_param_layout", "zero_shard_numel", "ZeroAdamW", "ZeroError", "ZeroLayout", "load", "zero_abi_version",
    "zero_adamw_shard_step", "zero_all_gather", "zero_device_status", "zero_flat_layout",
    "zero_flatten",
    "zero_last_error", "zero_reduce_scatter", "zero_selftest_wait_timeout",
    "zero_shard_segments", "zero_step", "zero_step_units", "zero_step_units_clip",
    "zero_clip_workspace_bytes", "zero_step_units_clip_noalloc",
    "zero_unflatten", "zero_step_units_host", "HostTables", "ZERO_HOST_GRADS_FREE", "ZERO_HOST_SM_COPY",
]
