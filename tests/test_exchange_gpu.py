"""GPU parity of the pack / unpack calls and of the multi-rank path, emulated on one GPU.

- ``reshard_execute_pack`` then ``reshard_execute_unpack`` with caller-owned message buffers
  (one buffer, or two with a device copy between them standing in for a transport) must give
  the oracle's destinations byte for byte, MXFP8 scales included.
- Several ranks of a process group are emulated in one process: each rank's partitioned plan
  packs with only its own pointers (every other rank's entry is NULL, so a table that named one
  would be refused on the host), ``exchange.loopback_transfers`` plays both transfer phases as
  device copies in posting order, and each rank unpacks. The union of all ranks' destinations
  must equal the oracle's, for colocated and disjoint placements, striped or not, MXFP8 and
  transposed layouts included. The kernels are the ones a multi-GPU run launches; only the wire
  is replaced by copies (kernels of different ranks never wait on each other).
"""
import numpy as np
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dtensor_resharding_gb300 as R
    from dtensor_resharding_gb300 import exchange
    from harness import assert_matches_oracle

CASES = {
    "dense_ragged": lambda: S.dense_ffn(layers=2, hidden=256, ffn=1000),
    "moe_ep16_to_ep8": lambda: S.moe_experts(layers=1, experts=32, hidden=256, ffn=96, dst="ep8"),
    "moe_tp4_mxfp8": lambda: S.moe_experts(layers=1, experts=16, hidden=256, ffn=256, dst="tp4"),
    "mesh2x4_to_3x2": lambda: S.mesh2d_to_1d(rows=143, cols=409, variant="2d"),
    "transposed_dst": lambda: S.transposed(shape=(1100, 640), src_mesh=(2,), src_pl=("S1",), dst_mesh=(3,),
                                           dst_pl=("S0",)),
    "many_small": lambda: S.many_small(n=60),
    "broadcast_8_replicas": lambda: _one((300, 520), (2,), ("S0",), (8,), ("R",)),
}


def _one(shape, sm, sp, dm, dp):
    ns, nd = int(np.prod(sm)), int(np.prod(dm))
    t = S.TensorDesc("w", shape, "bf16", sm, sp, dm, dp, [S.View(i) for i in range(ns)],
                     [S.View(i) for i in range(nd)], seed=19)
    return S.workloads._size_buffers(S.Workload("one", [t]), ns, nd)


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


@pytest.mark.parametrize("two_buffers", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_pack_unpack_with_caller_buffers(name, two_buffers):
    wl = CASES[name]()
    lay = _prepared(wl, misalign=2 if name == "many_small" else 0)
    plan = R.plan_workload(wl)
    st = R.reshard_plan_stats(plan)
    sp, dp = R.workload_pointers(wl, lay)
    stream = torch.cuda.current_stream().cuda_stream
    send = torch.empty(st["message_bytes"], dtype=torch.uint8, device="cuda")
    recv = torch.empty(st["recv_bytes"], dtype=torch.uint8, device="cuda") if two_buffers else send
    R.reshard_execute_pack(plan, sp, None, send, stream=stream)
    if two_buffers:
        recv.copy_(send)
    R.reshard_execute_unpack(plan, recv, dp, quant=wl.quant, stream=stream)
    torch.cuda.synchronize()
    assert R.reshard_plan_status(plan) == 0
    assert_matches_oracle(wl, lay)


def _owners(wl, layout, world):
    if layout == "random":
        rng = np.random.Generator(np.random.PCG64(len(wl.tensors) * 7919 + world))
        ns, nd = sum(t.n_src for t in wl.tensors), sum(t.n_dst for t in wl.tensors)
        return [int(x) for x in rng.integers(0, world, ns)], [int(x) for x in rng.integers(0, world, nd)]
    so, do = [], []
    for t in wl.tensors:
        so += [i % world if layout == "colocated" else i % max(1, world // 2) for i in range(t.n_src)]
        do += [j % world if layout == "colocated" else world // 2 + j % (world - world // 2) for j in range(t.n_dst)]
    return so, do


def _local(ptrs, owner, rank, per=1):
    out = np.array(ptrs, dtype=np.uint64).copy()
    for i, o in enumerate(owner):
        if o != rank:
            out[per * i: per * i + per] = 0
    return out


def _emulate(wl, world, layout, striped, misalign=0):
    lay = _prepared(wl, misalign)
    plan = R.plan_workload(wl)
    so, do = _owners(wl, layout, world)
    sp, dp = R.workload_pointers(wl, lay)
    per = 2 if wl.quant == "mxfp8" else 1
    stream = torch.cuda.current_stream().cuda_stream
    plans, sends, recvs = [], [], []
    for r in range(world):
        rp = R.reshard_plan_partition(plan, so, do, world, r, striped)
        st = R.reshard_plan_stats(rp)
        plans.append(rp)
        sends.append(torch.empty(max(16, st["message_bytes"]), dtype=torch.uint8, device="cuda"))
        recvs.append(torch.empty(max(16, st["recv_bytes"]), dtype=torch.uint8, device="cuda"))
        R.reshard_execute_pack(rp, _local(sp, so, r), _local(dp, do, r, per), sends[r], quant=wl.quant, stream=stream)
    moved = exchange.loopback_transfers(plans, sends, recvs)
    for r in range(world):
        R.reshard_execute_unpack(plans[r], recvs[r], _local(dp, do, r, per), quant=wl.quant, stream=stream)
    torch.cuda.synchronize()
    assert all(R.reshard_plan_status(p) == 0 for p in plans)
    assert_matches_oracle(wl, lay)
    sent = sum(R.reshard_plan_stats(p)["sent_bytes"] + R.reshard_plan_stats(p)["forwarded_bytes"] for p in plans)
    assert moved == sent


@pytest.mark.parametrize("striped", [True, False])
@pytest.mark.parametrize("layout", ["colocated", "disjoint"])
@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("name", sorted(CASES))
def test_ranks_emulated_on_one_gpu(name, world, layout, striped):
    _emulate(CASES[name](), world, layout, striped)


def test_fuzzed_layouts_random_owners_three_ranks():
    """Random shapes, meshes, dtypes and per-rank layouts with every pointer on a random one of
    three emulated ranks; buffers shifted by 8 bytes for every other case."""
    for i, wl in enumerate(S.fuzz_cases(40, seed=31)):
        _emulate(wl, 3, "random", i % 2 == 0, misalign=8 * (i % 2))


def test_exchange_through_a_one_rank_nccl_group():
    """exchange.reshard_exchange through a real NCCL process group of one rank (the one GPU):
    every region is a local copy made by the pack call, the group's first-exchange barrier goes
    through NCCL, and the result equals the oracle's. A second partition with the same plan and
    owners reuses the group without a barrier."""
    import os
    import socket
    import torch.distributed as dist
    if dist.is_initialized():
        pytest.skip("a process group already exists in this process")
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        for wl in (CASES["dense_ragged"](), CASES["moe_tp4_mxfp8"]()):
            lay = _prepared(wl)
            plan = R.plan_workload(wl)
            part = R.reshard_plan_partition(plan, [0] * plan.n_src_ptrs, [0] * plan.n_dst_ptrs, 1, 0, True)
            st = R.reshard_plan_stats(part)
            assert st["transfers"] == 0 and st["local_bytes"] == R.reshard_plan_stats(plan)["bytes_read"]
            send = torch.empty(16, dtype=torch.uint8, device="cuda")
            recv = torch.empty(16, dtype=torch.uint8, device="cuda")
            sp, dp = R.workload_pointers(wl, lay)
            exchange.reshard_exchange(part, sp, dp, send, recv, quant=wl.quant)
            torch.cuda.synchronize()
            assert_matches_oracle(wl, lay)
    finally:
        dist.destroy_process_group()
