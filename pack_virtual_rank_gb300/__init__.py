"""GB300-native sharded relay collectives on one GPU.

A relay collective runs among A active virtual ranks of an R-rank node and recruits
the H = R - A idle ranks as relay helpers (page "Link-balance the sharded relay
schedules (up to 3.2x vs NCCL)", torchrec pull request #4570). Every virtual rank's
buffers live in this GPU's HBM; the schedule's transfers and reductions run as
batched CUDA kernels (``csrc/``) behind the C ABI in ``include/relay.h``.
"""
from ._binding import (  # noqa: F401
    ALL_GATHER, ALL_TO_ALL, ALLREDUCE, ERR_CUDA, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, OK, BF16, COLLECTIVES, ESIZE, F32, FLAG_CHECK_HAZARDS, FLAG_DRY_RUN, FLAG_FUSED_PASSES, FLAG_SEPARATE_PASSES,
    FLAG_PAYLOAD_PARTIAL, FLAG_CHAINED, FLAG_KEEP_SCRATCH, I32, last_launch, device_status,
    KIND_DIRECT, KIND_LEGACY, KIND_RELAY, KIND_ZERO_CHUNK, PASS_NAMES, REDUCE_SCATTER,
    SCHEDULE_AUTO, SCHEDULE_DIRECT, SCHEDULE_LEGACY, SCHEDULE_RELAY, LIB_PATH, RelayError,
    RelayOpts, RelayPassInfo, RelayPlan, alloc_scratch, dtype_code, lib, make_opts,
    relay_all_gather, relay_all_to_all, relay_allreduce, relay_pass_name,
    relay_passthrough_helper_size, relay_plan, relay_plan_cost_bytes, relay_plan_link_bytes,
    relay_plan_passes, relay_reduce_scatter, group_ranks, relay_multi_group,
    relay_multi_group_link_bytes, alloc_multi_scratch, relay_pack_flat, relay_unpack_flat,
    relay_allreduce_noalloc, relay_helper_size, relay_active_scratch_size,
    relay_helper_contract_size, relay_copy)
