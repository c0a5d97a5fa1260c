"""GB300-native DTensor -> DTensor reshard executor (single GPU, sm_103a).

The public calls mirror the C ABI in include/reshard.h:
``reshard_plan_create``, ``reshard_plan_batch``, ``reshard_execute``, ``reshard_execute_pack`` /
``reshard_execute_unpack``, ``reshard_plan_partition`` / ``reshard_plan_transfers`` (the multi-process
exchange, driven by ``exchange``), ``reshard_plan_stats``, ``reshard_plan_regions``,
``reshard_plan_group_members``, ``reshard_plan_destroy``, ``reshard_last_error``. Importing the
package loads libreshard.so and raises if it is not built.
"""
from .binding import (  # noqa: F401
    Plan, ReshardError, Spec, View, LIB_PATH, EXPORTED, STATS_FIELDS, pointer_array,
    reshard_plan_create, reshard_plan_batch, reshard_plan_blockwise_fp8, reshard_execute, reshard_execute_pack, reshard_execute_unpack,
    reshard_plan_partition, reshard_plan_transfers, reshard_execute_static, reshard_plan_stats, reshard_plan_regions,
    reshard_plan_group_members, reshard_plan_items, reshard_plan_slabs, reshard_plan_status,
    reshard_plan_destroy, reshard_last_error, make_spec,
    RESHARD_OK, RESHARD_ERR_INVALID_ARG, RESHARD_ERR_UNSUPPORTED, RESHARD_ERR_CUDA, RESHARD_ERR_OOM,
    RESHARD_ERR_COVERAGE, RESHARD_DIRECT, RESHARD_PACKED, RESHARD_QUANT_NONE, RESHARD_QUANT_MXFP8,
    RESHARD_STRIPED, RESHARD_SEND, RESHARD_RECV, RESHARD_SEND_BUF, RESHARD_RECV_BUF,
)
from .workload import plan_workload, workload_pointers  # noqa: F401
