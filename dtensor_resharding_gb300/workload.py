"""Plan and pointer marshalling for a whole workload description (duck-typed).

A workload object has ``tensors`` (each with global_shape, dtype, meshes, placements and
per-rank views carrying .buffer/.offset/.strides), ``src_buffer_numel`` / ``dst_buffer_numel``
(capacities for the bounds check) and ``quant``. A layout object maps buffers to device
pointers through ``src_ptrs(wl, t)`` / ``dst_ptrs(wl, t)``.
"""
from __future__ import annotations

from .binding import Plan, pointer_array, reshard_plan_batch, reshard_plan_blockwise_fp8


def plan_workload(wl) -> Plan:
    """One batched plan over every tensor of the workload (view capacities bound-checked)."""
    src_cap = [[wl.src_buffer_numel[v.buffer] for v in t.src_views] for t in wl.tensors]
    dst_cap = [[wl.dst_buffer_numel[v.buffer] for v in t.dst_views] for t in wl.tensors]
    block = getattr(wl, "block", None)
    if block:
        # blockwise FP8: the first half of the tensors are the weights, the second their scales
        n = len(wl.tensors) // 2
        return reshard_plan_blockwise_fp8(wl.tensors[:n], block, src_cap[:n], dst_cap[:n])
    return reshard_plan_batch(wl.tensors, src_cap, dst_cap)


def workload_pointers(wl, layout):
    """Flat source / destination pointer arrays in plan order (uint64 numpy arrays)."""
    src, dst = [], []
    for t in range(len(wl.tensors)):
        src += layout.src_ptrs(wl, t)
        dst += layout.dst_ptrs(wl, t)
    return pointer_array(src), pointer_array(dst)
