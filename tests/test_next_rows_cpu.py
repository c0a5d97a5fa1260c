"""Workloads beyond the headline rows, on the CPU: KV heads below TP, vLLM fused w13, per-expert
sources, blockwise FP8 with scales. Plans against the oracle, and the item tables emulated."""
import numpy as np
import pytest

import dtensor_resharding_gb300 as R
import synthetic as S
from oracle import golden as G

from test_items_cpu import check_bounds, check_transpose_bounds, emulate, _oracle
from test_parity_gpu import SMALL

NEXT = [k for k in SMALL if k.startswith(("qkv_", "moe_w13", "moe_fp8"))]


def _planner_regions(plan):
    return sorted((t, tuple(R.reshard_plan_group_members(plan, g)), s, box)
                  for t, s, g, box in R.reshard_plan_regions(plan))


@pytest.mark.parametrize("name", NEXT)
def test_next_rows_plan_matches_oracle_regions(name):
    wl = SMALL[name]()
    plan = R.plan_workload(wl)
    got = _planner_regions(plan)
    for ti, t in enumerate(wl.tensors):
        nd = len(t.global_shape)
        mine = sorted((m, s, box[:nd]) for tt, m, s, box in got if tt == ti)
        assert mine == G.source_regions(t), (name, t.name)


@pytest.mark.parametrize("mode", ["direct", "packed"])
@pytest.mark.parametrize("name", NEXT)
def test_next_rows_item_tables_reproduce_oracle(name, mode):
    wl = SMALL[name]()
    lay = S.allocate(wl, "cpu")
    S.fill_sources(wl, lay)
    plan = R.plan_workload(wl)
    for which in (0, 1, 2):
        check_bounds(wl, lay, plan, which)
        check_transpose_bounds(wl, lay, plan, which)
    assert np.array_equal(emulate(wl, lay, plan, mode), _oracle(wl, lay))


def test_kv_heads_below_tp_replicate_inside_groups():
    """Q=16 heads, KV=2, TP8: each KV head lives on 4 ranks; the plan reads each once."""
    wl = S.qkv_kv_below_tp(layers=1, q_heads=16, kv_heads=2, head_dim=16, hidden=96)
    st = R.reshard_plan_stats(R.plan_workload(wl))
    k_bytes = 2 * 16 * 96 * 2
    q_bytes = 16 * 16 * 96 * 2
    assert st["bytes_read"] == q_bytes + 2 * k_bytes
    assert st["bytes_written"] == q_bytes + 2 * 4 * k_bytes


def test_blockwise_fp8_scales_follow_their_blocks():
    """Every destination's scale shard covers exactly the blocks of its weight shard."""
    wl = SMALL["moe_fp8_blockwise"]()
    n = len(wl.tensors) // 2
    for w, sc in zip(wl.tensors[:n], wl.tensors[n:]):
        for mesh, pls in ((w.src_mesh, w.src_placements), (w.dst_mesh, w.dst_placements)):
            for coord in G.mesh_coords(mesh):
                wb = G.shard_box(w.global_shape, mesh, pls, coord)
                sb = G.shard_box(sc.global_shape, mesh, pls, coord)
                for d, b in ((-2, wl.block[0]), (-1, wl.block[1])):
                    assert sb[d][0] == wb[d][0] // b and sb[d][1] == -(-wb[d][1] // b)


def test_blockwise_fp8_rejects_off_grid_splits():
    bad = S.moe_fp8_blockwise(layers=1, experts=4, hidden=256, ffn=1000, ep_src=2, dp_src=1, tp_dst=3, dp_dst=1)
    with pytest.raises(R.ReshardError) as e:
        R.plan_workload(bad)
    assert e.value.code == R.RESHARD_ERR_UNSUPPORTED and "block grid" in str(e.value)
