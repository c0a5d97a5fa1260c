"""Plan lifetime on the GPU: destroy waits for the plan's own executes (an event per stream it
used), never for the whole device, and never invalidates a stream capture in progress."""
import gc

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


@pytest.fixture(autouse=True)
def _cleanup():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_plan_dropped_while_executes_on_two_streams_are_queued():
    """Executes on stream A, then on stream B ordered after A; the handle is collected at once.
    destroy waits for both streams' last executes, so both results are complete."""
    wl = S.dense_ffn(layers=2, hidden=256, ffn=1000)
    lay_a, lay_b = _prepared(wl), _prepared(wl, misalign=2)
    plan = R.plan_workload(wl)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    pa, da = R.workload_pointers(wl, lay_a)
    pb, db = R.workload_pointers(wl, lay_b)
    R.reshard_execute(plan, pa, da, stream=sa.cuda_stream)
    ev = torch.cuda.Event()
    ev.record(sa)
    sb.wait_event(ev)
    R.reshard_execute(plan, pb, db, mode="packed", stream=sb.cuda_stream)
    del plan
    gc.collect()
    torch.cuda.synchronize()
    assert_matches_oracle(wl, lay_a)
    assert_matches_oracle(wl, lay_b)


def test_two_plans_run_concurrently_on_two_streams():
    w1 = S.moe_experts(layers=1, experts=32, hidden=256, ffn=96, dst="ep8")
    w2 = S.mesh2d_to_1d(rows=1434, cols=4096, variant="2d")
    l1, l2 = _prepared(w1), _prepared(w2)
    p1, p2 = R.plan_workload(w1), R.plan_workload(w2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    a1, b1 = R.workload_pointers(w1, l1)
    a2, b2 = R.workload_pointers(w2, l2)
    for _ in range(3):
        R.reshard_execute(p1, a1, b1, stream=s1.cuda_stream)
        R.reshard_execute(p2, a2, b2, stream=s2.cuda_stream)
    torch.cuda.synchronize()
    assert R.reshard_plan_status(p1) == 0 and R.reshard_plan_status(p2) == 0
    assert_matches_oracle(w1, l1)
    assert_matches_oracle(w2, l2)


def test_destroy_during_another_plans_stream_capture():
    """A plan destroyed while another plan's execute is being captured into a CUDA graph: the
    destroy's waits and frees run in relaxed capture mode, so the capture stays valid, and the
    graph replays to the oracle's result."""
    w_cap = S.dense_ffn(layers=1, hidden=256, ffn=1024)
    w_old = S.uneven_tp(rows=1433, cols=409)
    lay = _prepared(w_cap)
    old_lay = _prepared(w_old)
    cap_plan = R.plan_workload(w_cap)
    old_plan = R.plan_workload(w_old)
    sp, dp = R.workload_pointers(w_cap, lay)
    R.reshard_execute(cap_plan, sp, dp, stream=torch.cuda.current_stream().cuda_stream)   # binds, uploads
    op, od = R.workload_pointers(w_old, old_lay)
    R.reshard_execute(old_plan, op, od, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert_matches_oracle(w_old, old_lay)
    S.fill_canary(lay)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        R.reshard_execute(cap_plan, sp, dp, stream=s.cuda_stream)
        R.reshard_plan_destroy(old_plan)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert_matches_oracle(w_cap, lay)
    del g
    R.reshard_plan_destroy(cap_plan)   # after the graph that captured its execute is gone
