"""Seeded synthetic workloads shared by the tests, the bench and the oracle's callers.

This package holds problem descriptions (global shapes, meshes, placements, buffer views)
and seeded value generators only. It contains none of the reshard method's arithmetic.
"""
from .workloads import (  # noqa: F401
    View, TensorDesc, Workload, Layout,
    example_8x8, dense_ffn, moe_experts, uneven_tp, mesh2d_to_1d, many_small, transposed, qkv_kv_below_tp, moe_w13, moe_fp8_blockwise,
    large_offsets,
    brute_force_cases, fuzz_cases,
    workload_by_name, WORKLOAD_NAMES,
    local_shape, allocate, fill_sources, fill_canary, DTYPES,
)
