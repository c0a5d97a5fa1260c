"""reshard_execute_static: the reshard for callers that cannot let a library allocate GPU memory.

Such callers (an inference engine that keeps almost all device memory reserved for its KV
cache, a framework whose own allocator owns the device heap) cannot accept a cudaMalloc in the
middle of a refit: it can fail for lack of memory, and it synchronizes the device. This entry
point keeps its descriptor tables in a fixed array inside the library instead. Its output must
be byte-identical (tolerance 0, as for every copy here) to reshard_execute's, on two calls in a
row with different plans, so that stale tables left by the first call cannot leak into the
second. Collected last, and independent of any other test's state.
"""
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dtensor_resharding_gb300 as R


def _prepared(wl, misalign=0):
    lay = S.allocate(wl, "cuda", misalign=misalign)
    S.fill_sources(wl, lay)
    S.fill_canary(lay)
    return lay


def test_static_entry_matches_execute_on_two_calls_in_a_row():
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
        for t in range(len(wl.tensors)):
            es = S.DTYPES[wl.tensors[t].dtype][1]
            for v in wl.tensors[t].dst_views:
                n = wl.dst_buffer_numel[v.buffer] * es
                x = a.dst_slab[a.dst_off[v.buffer]: a.dst_off[v.buffer] + n]
                y = b.dst_slab[b.dst_off[v.buffer]: b.dst_off[v.buffer] + n]
                assert torch.equal(x, y), (wl.name, t, v.buffer)


def test_static_entry_rejects_plans_beyond_its_array():
    # 640 x 640 regions: 409,600 work items of 64 bytes, more than the fixed array holds
    d = S.TensorDesc("w", (640, 1280), "i32", (640,), ("S0",), (640,), ("S1",),
                     [S.View(i) for i in range(640)], [S.View(i) for i in range(640)])
    plan = R.reshard_plan_create(d)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute_static(plan, [1] * 640, [1] * 640)
    assert e.value.code == R.RESHARD_ERR_UNSUPPORTED and "at most" in str(e.value)
