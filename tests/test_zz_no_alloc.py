"""reshard_execute_static: the reshard for callers that cannot let a library allocate GPU memory.

Such callers (an inference engine that keeps almost all device memory reserved for its KV
cache, a framework whose own allocator owns the device heap) cannot accept a cudaMalloc in the
middle of a refit: it can fail for lack of memory, and it synchronizes the device. This entry
point keeps its descriptor tables in a fixed array inside the library instead. Its output must
equal the oracle's byte for byte (tolerance 0, as for every copy here) and reshard_execute's, on
two calls in a row with different plans, so that stale tables left by the first call cannot
leak into the second. Collected last, and independent of any other test's state.
"""
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dtensor_resharding_gb300 as R
    from harness import assert_matches_oracle


def _prepared(wl, misalign=0):
    lay = S.allocate(wl, "cuda", misalign=misalign)
    S.fill_sources(wl, lay)
    S.fill_canary(lay)
    return lay


def test_static_entry_matches_oracle_and_execute_on_two_calls_in_a_row():
    workloads = [S.dense_ffn(layers=2, hidden=256, ffn=1000),
                 S.mesh2d_to_1d(rows=143, cols=409, variant="2d")]
    plans = [R.plan_workload(wl) for wl in workloads]
    stream = torch.cuda.current_stream().cuda_stream
    # reference output through the existing entry point
    want = []
    for wl, plan in zip(workloads, plans):
        lay = _prepared(wl)
        sp, dp = R.workload_pointers(wl, lay)
        R.reshard_execute(plan, sp, dp, stream=stream)
        want.append(lay)
    # the allocation-free entry point, two calls back to back on one stream, different plans
    got = []
    for wl, plan, mis in zip(workloads, plans, (0, 2)):
        lay = _prepared(wl, misalign=mis)
        sp, dp = R.workload_pointers(wl, lay)
        R.reshard_execute_static(plan, sp, dp, stream=stream)
        got.append(lay)
    torch.cuda.synchronize()
    for wl, a, b in zip(workloads, want, got):
        assert_matches_oracle(wl, b)
        for t in range(len(wl.tensors)):
            es = S.DTYPES[wl.tensors[t].dtype][1]
            for v in wl.tensors[t].dst_views:
                n = wl.dst_buffer_numel[v.buffer] * es
                x = a.dst_slab[a.dst_off[v.buffer]: a.dst_off[v.buffer] + n]
                y = b.dst_slab[b.dst_off[v.buffer]: b.dst_off[v.buffer] + n]
                assert torch.equal(x, y), (wl.name, t, v.buffer)


def test_static_entry_refuses_pageable_memory_before_any_launch():
    """The pointers are checked like reshard_execute's: pageable host memory is refused on the
    host instead of reaching a kernel."""
    import dataclasses
    wl = S.dense_ffn(layers=1, hidden=256, ffn=1000)
    lay = _prepared(wl)
    plan = R.plan_workload(wl)
    pageable = torch.empty(lay.src_slab.numel(), dtype=torch.uint8)
    sp, dp = R.workload_pointers(wl, dataclasses.replace(lay, src_slab=pageable))
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute_static(plan, sp, dp)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "pageable" in str(e.value)
    sp, dp = R.workload_pointers(wl, lay)
    R.reshard_execute_static(plan, sp, dp, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert_matches_oracle(wl, lay)
