"""The C ABI on the host (no GPU): exported symbols, the planner against the oracle, validation."""
import os
import re

import numpy as np
import pytest

import dtensor_resharding_gb300 as R
import synthetic as S
from oracle import golden as G

from conftest import ROOT, read_fixture


def test_library_exports_every_declared_symbol():
    hdr = open(os.path.join(ROOT, "include", "reshard.h")).read()
    declared = set(re.findall(r"^(?:int|const char \*)\s*(reshard_\w+)\(", hdr, flags=re.M))
    assert declared == set(R.EXPORTED)
    for name in declared:
        assert hasattr(R.binding.LIB, name)
        assert callable(getattr(R, name))


def _planner_regions(plan):
    out = []
    for t, s, g, box in R.reshard_plan_regions(plan):
        members = tuple(R.reshard_plan_group_members(plan, g))
        out.append((t, members, s, box))
    return out


def test_planner_8x8_example_regions():
    rows, _ = read_fixture("example_8x8.txt")
    want = sorted(((int(d),), int(s), ((int(r0), int(r1)), (int(c0), int(c1)))) for d, s, r0, r1, c0, c1 in rows)
    plan = R.plan_workload(S.example_8x8())
    got = sorted((m, s, box[:2]) for _, m, s, box in _planner_regions(plan))
    assert got == want
    st = R.reshard_plan_stats(plan)
    assert st["regions"] == 8 and st["bytes_read"] == 128 and st["bytes_written"] == 128


def test_planner_tp4_to_tp2dp2_replicas():
    rows, meta = read_fixture("tp4_to_tp2dp2.txt")
    want = sorted((tuple(int(x) for x in g.split(",")), int(s), ((int(r0), int(r1)), (int(c0), int(c1))))
                  for g, s, r0, r1, c0, c1 in rows)
    d = S.TensorDesc("w", (8, 4), "i32", (4,), ("S0",), (2, 2), ("R", "S0"),
                     [S.View(i) for i in range(4)], [S.View(i) for i in range(4)])
    plan = R.reshard_plan_create(d)
    got = sorted((m, s, box[:2]) for _, m, s, box in _planner_regions(plan))
    assert got == want
    st = R.reshard_plan_stats(plan)
    assert st["bytes_read"] == int(meta["bytes_read"][0])
    assert st["bytes_written"] == int(meta["bytes_written"][0])


def test_planner_matches_oracle_brute_force():
    """Regions, chosen sources and replica groups equal the oracle's element-wise enumeration."""
    for wl in S.brute_force_cases(250, seed=31):
        t = wl.tensors[0]
        plan = R.plan_workload(wl)
        nd = len(t.global_shape)
        got = sorted((m, s, box[:nd]) for _, m, s, box in _planner_regions(plan))
        assert got == G.source_regions(t), (t.global_shape, t.src_mesh, t.src_placements, t.dst_mesh, t.dst_placements)
        st = R.reshard_plan_stats(plan)
        acc = G.byte_accounting(t)
        assert st["bytes_read"] == acc["bytes_read"]
        assert st["bytes_written"] == acc["bytes_written"]
        assert st["gather_bcast_bytes"] == acc["gather_bcast_bytes"]
        assert st["dst_groups"] == acc["dst_groups"]


@pytest.mark.parametrize("name", ["dense_ffn_32x14336x4096_tp8_to_dp2tp2", "moe_8x128x1536x4096_ep16_to_ep8",
                                  "moe_8x128x1536x4096_ep16_to_tp4_mxfp8", "uneven_14336x4096_tp6_to_tp5",
                                  "mesh2x4_to_3_14336x4096", "mesh2x4_to_3x2_14336x4096"])
def test_full_size_byte_accounting(name):
    wl = S.workload_by_name(name)
    plan = R.plan_workload(wl)
    st = R.reshard_plan_stats(plan)
    acc = [G.byte_accounting(t) for t in wl.tensors]
    assert st["bytes_read"] == sum(a["bytes_read"] for a in acc)
    assert st["bytes_written"] == sum(a["bytes_written"] for a in acc)
    total = sum(int(np.prod(t.global_shape)) * G.ESIZE[t.dtype] for t in wl.tensors)
    assert st["global_bytes"] == total and st["gather_bcast_bytes"] == 2 * total
    assert st["bytes_read"] == total  # each element read once per destination replica group


def test_dense_ffn_plan_shape():
    st = R.reshard_plan_stats(R.plan_workload(S.dense_ffn()))
    # 32 layers x 3 projections x 8 source ranks; each source shard lies inside one TP2 shard
    assert st["regions"] == 768 and st["dst_groups"] == 192 and st["messages"] == 8
    assert st["bytes_read"] == 11_274_289_152 and st["bytes_written"] == 22_548_578_304


def test_validation_lists_every_violation():
    d = S.TensorDesc("w", (8, -1), "bf16", (2,), ("S2",), (0,), ("S1",),
                     [S.View(0), S.View(1)], [S.View(0)])
    with pytest.raises(R.ReshardError) as e:
        R.reshard_plan_create(d)
    msg = str(e.value)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG
    assert "global_shape[1] < 0" in msg and "dst_mesh.shape[0] < 1" in msg


def test_validation_batch_lists_all_tensors():
    good = S.TensorDesc("a", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",), [S.View(0)] * 2, [S.View(0)] * 4)
    bad1 = S.TensorDesc("b", (8, 8), "bf16", (2,), ("S5",), (4,), ("S1",), [S.View(0)] * 2, [S.View(0)] * 4)
    bad2 = S.TensorDesc("c", (8, 8), "nope", (2,), ("S0",), (4,), ("S1",), [S.View(0)] * 2, [S.View(0)] * 4)
    bad2.dtype = 99
    with pytest.raises(R.ReshardError) as e:
        R.reshard_plan_batch([good, bad1, bad2])
    msg = str(e.value)
    assert "tensor 1:" in msg and "tensor 2:" in msg and "tensor 0:" not in msg


def test_view_capacity_overflow():
    d = S.TensorDesc("w", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",),
                     [S.View(0, 0), S.View(1, 10)], [S.View(i) for i in range(4)])
    with pytest.raises(R.ReshardError) as e:
        R.reshard_plan_create(d, src_capacity=[32, 32], dst_capacity=[16] * 4)
    assert "overflows its buffer" in str(e.value)


def test_destination_views_whose_elements_alias_are_refused():
    """A destination view that maps two elements to one offset (a row pitch shorter than its
    rows, a zero stride) is refused with the view named; the same strides on a source view (read
    only) plan, and so do padded, transposed and interleaved destination strides."""
    for strides in ((1, 1), (0, 1), (1, 2)):        # local shape (8, 2): rows overlap
        bad = S.TensorDesc("w", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",), [S.View(0), S.View(1)],
                           [S.View(0, 0, strides)] + [S.View(i) for i in range(1, 4)])
        with pytest.raises(R.ReshardError) as e:
            R.reshard_plan_create(bad)
        assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "dst view 0 maps two elements to one offset" in str(e.value)
    src_alias = S.TensorDesc("w", (8, 8), "bf16", (1,), ("R",), (4,), ("S1",), [S.View(0, 0, (0, 1))],
                             [S.View(i) for i in range(4)])
    R.reshard_plan_create(src_alias)                # every row of the source reads one buffer row
    for strides in ((3, 1), (1, 8), (4, 1)):        # padded rows, column-major, rows two apart
        ok = S.TensorDesc("w", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",), [S.View(0), S.View(1)],
                          [S.View(0, 0, strides)] + [S.View(i) for i in range(1, 4)])
        R.reshard_plan_create(ok)


def test_negative_stride_rejected_and_transposed_view_planned():
    bad = S.TensorDesc("w", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",),
                       [S.View(0, 0, (8, -1)), S.View(1)], [S.View(i) for i in range(4)])
    with pytest.raises(R.ReshardError) as e:
        R.reshard_plan_create(bad)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG
    wl = S.transposed(shape=(300, 200), src_mesh=(2,), src_pl=("S0",), dst_mesh=(2,), dst_pl=("S1",))
    plan = R.plan_workload(wl)
    t, *_ = R.reshard_plan_items(plan, 3)
    assert len(t) > 0 and len(R.reshard_plan_items(plan, 0)[0]) == 0
    slabs = R.reshard_plan_slabs(plan)
    # direct: one slab per source shard; unpack: one per message region (2 x 2 regions)
    assert len(set(t["slab"])) == 2 and len(slabs) == 6 and all(sl[1] == 2 for sl in slabs)


def test_mesh_rank_permutation():
    d = S.TensorDesc("w", (8, 8), "i32", (2,), ("S0",), (4,), ("S1",), [S.View(0), S.View(1)],
                     [S.View(i) for i in range(4)])
    d.dst_ranks = [3, 2, 1, 0]
    plan = R.reshard_plan_create(d)
    regs = _planner_regions(plan)
    # destination pointer 3 holds mesh position 0: columns 0..1
    assert sorted(box[1] for _, m, s, box in regs if m == (3,)) == [(0, 2), (0, 2)]
    d.dst_ranks = [0, 0, 1, 2]
    with pytest.raises(R.ReshardError):
        R.reshard_plan_create(d)


def test_execute_errors_before_touching_a_gpu():
    wl = S.dense_ffn(layers=1, hidden=64, ffn=100)   # last dims not multiples of 32 -> no MXFP8
    plan = R.plan_workload(wl)
    n_src = plan.n_src_ptrs
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute(plan, [1] * n_src, [1] * plan.n_dst_ptrs, quant="mxfp8")
    assert e.value.code == R.RESHARD_ERR_UNSUPPORTED
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute(plan, [0] * n_src, [1] * plan.n_dst_ptrs)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "NULL" in str(e.value)
    with pytest.raises(R.ReshardError):
        R.reshard_execute(plan, [1] * n_src, [1] * plan.n_dst_ptrs, mode=7)


def test_mxfp8_region_edges_must_hold_whole_blocks():
    # source splits the last dim at 48 (not a multiple of 32): blocks would straddle sources
    d = S.TensorDesc("w", (4, 96), "bf16", (2,), ("S1",), (1,), ("R",), [S.View(0), S.View(1)], [S.View(0)])
    plan = R.reshard_plan_create(d)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute(plan, [1, 1], [1, 1], quant="mxfp8")
    assert "straddle" in str(e.value)


def test_empty_batch_and_empty_tensor():
    plan = R.reshard_plan_batch([])
    assert R.reshard_plan_stats(plan)["regions"] == 0
    R.reshard_execute(plan, [], [])
    d = S.TensorDesc("w", (0, 8), "bf16", (2,), ("S0",), (4,), ("S1",), [S.View(0), S.View(1)],
                     [S.View(i) for i in range(4)])
    plan = R.reshard_plan_create(d)
    assert R.reshard_plan_stats(plan)["regions"] == 0
    R.reshard_execute(plan, [0, 0], [0] * 4)


def test_static_entry_rejects_transposing_plans_before_any_cuda_call():
    wl = S.transposed(shape=(300, 200), src_mesh=(2,), src_pl=("S0",), dst_mesh=(2,), dst_pl=("S1",))
    plan = R.plan_workload(wl)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute_static(plan, [1] * plan.n_src_ptrs, [1] * plan.n_dst_ptrs)
    assert e.value.code == R.RESHARD_ERR_UNSUPPORTED and "transposing" in str(e.value)


def test_static_entry_rejects_plans_beyond_its_array_before_any_cuda_call():
    # 640 x 640 regions: 409,600 work items of 64 bytes, more than the fixed array holds; the
    # size check comes first, so the (fabricated) pointers are never looked at
    d = S.TensorDesc("w", (640, 1280), "i32", (640,), ("S0",), (640,), ("S1",),
                     [S.View(i) for i in range(640)], [S.View(i) for i in range(640)])
    plan = R.reshard_plan_create(d)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute_static(plan, [1] * 640, [1] * 640)
    assert e.value.code == R.RESHARD_ERR_UNSUPPORTED and "at most" in str(e.value)


def test_pack_and_unpack_check_their_arguments_on_the_host():
    wl = S.dense_ffn(layers=1, hidden=64, ffn=100)
    plan = R.plan_workload(wl)
    ns, nd = plan.n_src_ptrs, plan.n_dst_ptrs
    for buf in (None, 8):   # missing, and not 16-byte aligned
        with pytest.raises(R.ReshardError) as e:
            R.reshard_execute_pack(plan, [1] * ns, None, buf)
        assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "send_buf" in str(e.value)
        with pytest.raises(R.ReshardError) as e:
            R.reshard_execute_unpack(plan, buf, [1] * nd)
        assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "recv_buf" in str(e.value)
    with pytest.raises(R.ReshardError) as e:   # an unpartitioned plan's pack copies, never quantizes
        R.reshard_execute_pack(plan, [1] * ns, None, 16, quant="mxfp8")
    assert e.value.code in (R.RESHARD_ERR_INVALID_ARG, R.RESHARD_ERR_UNSUPPORTED)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute_pack(plan, [0] * ns, None, 16)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "NULL" in str(e.value)
    st = R.reshard_plan_stats(plan)
    assert st["recv_bytes"] == st["message_bytes"] > 0 and st["rank"] == -1 and st["world"] == 0


def test_status_is_zero_before_any_execute():
    plan = R.plan_workload(S.example_8x8())
    assert R.reshard_plan_status(plan) == 0


def test_dp8_replicas_are_read_once():
    """The planner reads one of the eight DP replicas: naive per-replica reading moves 8x more."""
    _, meta = read_fixture("dp8_dedup.txt")
    d = S.TensorDesc("w", (4096, 2560), "bf16", (8, 2), ("R", "S0"), (4, 4), ("R", "S0"),
                     [S.View(i) for i in range(16)], [S.View(i) for i in range(16)])
    st = R.reshard_plan_stats(R.reshard_plan_create(d))
    total = 4096 * 2560 * 2
    assert st["bytes_read"] == total
    naive = int(meta["replicas_on_source"][0]) * total
    assert naive // st["bytes_read"] == int(meta["bytes_read_ratio_naive_over_planned"][0])
    assert st["bytes_written"] == 4 * total   # four engines, each a full TP4 copy
    # every region's source is the lowest-index replica (dp = 0): pointer indices 0 and 1
    assert {s for _, s, _, _ in R.reshard_plan_regions(R.reshard_plan_create(d))} == {0, 1}


def test_batch_marshalling_equals_single_tensor_plans():
    """The packed batch marshalling gives each tensor the same regions as planning it alone
    (views with offsets and strides, rank permutations, capacities)."""
    cases = list(S.fuzz_cases(40, seed=29))
    d = S.TensorDesc("p", (8, 8), "i32", (2,), ("S0",), (4,), ("S1",), [S.View(0), S.View(1)],
                     [S.View(i) for i in range(4)])
    d.dst_ranks = [3, 2, 1, 0]
    descs = [wl.tensors[0] for wl in cases] + [d]
    caps_s = [[wl.src_buffer_numel[v.buffer] for v in wl.tensors[0].src_views] for wl in cases] + [[64, 64]]
    caps_d = [[wl.dst_buffer_numel[v.buffer] for v in wl.tensors[0].dst_views] for wl in cases] + [[64] * 4]
    batch = R.reshard_plan_batch(descs, caps_s, caps_d)
    got = {}
    for t, m, s, box in _planner_regions(batch):
        got.setdefault(t, []).append((m, s, box))
    for t, desc in enumerate(descs):
        alone = R.reshard_plan_create(desc, caps_s[t], caps_d[t])
        want = sorted((m, s, box) for _, m, s, box in _planner_regions(alone))
        assert sorted(got.get(t, [])) == want, t
    st = R.reshard_plan_stats(batch)
    assert st["n_tensors"] == len(descs)


def test_every_entry_point_refuses_null_and_out_of_range_arguments():
    """NULL plans, NULL outputs and out-of-range indices return INVALID_ARG with a message, on the
    host, before any device work; nothing crashes."""
    import ctypes
    L = R.binding.LIB
    inv = R.RESHARD_ERR_INVALID_ARG
    n = ctypes.c_int64()
    st = R.binding.StatsT()
    i32 = ctypes.c_int32()
    assert L.reshard_plan_create(None, ctypes.byref(ctypes.c_void_p())) == inv
    assert L.reshard_plan_batch(None, 1, ctypes.byref(ctypes.c_void_p())) == inv
    assert L.reshard_plan_stats(None, ctypes.byref(st)) == inv
    assert L.reshard_plan_regions(None, 0, None, None, None, None, None, ctypes.byref(n)) == inv
    assert L.reshard_plan_slabs(None, 0, None, ctypes.byref(n)) == inv
    assert L.reshard_plan_status(None, ctypes.byref(i32), 0) == inv
    assert L.reshard_execute(None, None, None, 0, 0, None) == inv
    assert L.reshard_execute_static(None, None, None, None) == inv
    assert L.reshard_execute_pack(None, None, None, None, 0, None) == inv
    assert L.reshard_execute_unpack(None, None, None, 0, None) == inv
    assert L.reshard_plan_partition(None, None, None, 1, 0, 0, ctypes.byref(ctypes.c_void_p())) == inv
    assert L.reshard_plan_transfers(None, 1, 0, None, ctypes.byref(n)) == inv
    assert L.reshard_plan_destroy(None) == R.RESHARD_OK
    plan = R.plan_workload(S.example_8x8())
    assert L.reshard_plan_stats(plan.handle, None) == inv
    assert L.reshard_plan_group_members(plan.handle, 10 ** 6, 0, None, ctypes.byref(n)) == inv
    assert L.reshard_plan_group_members(plan.handle, -1, 0, None, ctypes.byref(n)) == inv
    assert L.reshard_plan_items(plan.handle, 9, 0, None, ctypes.byref(n), None, None, None, None, None) == inv
    assert L.reshard_plan_items(plan.handle, -1, 0, None, ctypes.byref(n), None, None, None, None, None) == inv
    assert L.reshard_plan_transfers(plan.handle, 3, 0, None, ctypes.byref(n)) == inv
    assert L.reshard_plan_partition(plan.handle, None, None, 1, 0, 0, None) == inv
    assert R.reshard_last_error()  # the last refusal left a message
    with pytest.raises(R.ReshardError):
        R.reshard_plan_group_members(plan, 10 ** 6)


def test_torch_placement_objects_are_accepted():
    """PyTorch's own DTensor placements (Shard(d), Replicate(), e.g. a model's
    DTensor.placements) plan exactly like their string spellings, in both marshalling paths."""
    from torch.distributed.tensor import Replicate, Shard
    a = S.TensorDesc("w", (12, 10), "bf16", (2, 2), ("S0", "R"), (4,), ("S1",),
                     [S.View(i) for i in range(4)], [S.View(i) for i in range(4)])
    b = S.TensorDesc("w", (12, 10), "bf16", (2, 2), (Shard(0), Replicate()), (4,), (Shard(1),),
                     [S.View(i) for i in range(4)], [S.View(i) for i in range(4)])
    want = sorted(_planner_regions(R.reshard_plan_create(a)))
    assert sorted(_planner_regions(R.reshard_plan_create(b))) == want
    assert sorted(_planner_regions(R.reshard_plan_batch([b]))) == want


def test_spec_containers_plan_like_workload_descriptions():
    """R.Spec / R.View (the binding's own containers) plan exactly like the test descriptions."""
    a = S.TensorDesc("w", (12, 10), "f32", (2,), ("S0",), (2, 2), ("R", "S1"),
                     [S.View(0), S.View(1)], [S.View(0, 3, (8, 1)), S.View(1, 0, (8, 1)),
                                              S.View(2, 0, (8, 1)), S.View(3, 0, (8, 1))])
    b = R.Spec((12, 10), "f32", (2,), ["S0"], (2, 2), ["R", "S1"],
               dst_views=[R.View(3, (8, 1)), R.View(0, (8, 1)), R.View(0, (8, 1)), R.View(0, (8, 1))])
    assert sorted(_planner_regions(R.reshard_plan_create(b))) == sorted(_planner_regions(R.reshard_plan_create(a)))
    st = R.reshard_plan_stats(R.reshard_plan_batch([b, b]))
    assert st["n_tensors"] == 2 and st["bytes_written"] == 2 * 2 * 12 * 10 * 4
