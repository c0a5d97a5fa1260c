"""The multi-process reshard on CPU: gloo ranks pack, exchange real message bytes, and unpack.

Every rank partitions the same plan for itself (``reshard_plan_partition``), runs its pack pass
(local copies and outgoing messages) and its unpack pass with a host emulation of the device
item tables, and moves the message bytes with ``exchange.run_transfers`` over a gloo process
group (world size 2 and 4). Checked against the oracle and the pages' accounting:
- every rank's destination buffers equal the oracle's shards byte for byte; sources held by
  other ranks are poisoned, so a rank that read one would be caught; destination buffers held
  by other ranks stay untouched;
- the transfers pair up across ranks (sizes and counts per peer and phase);
- each region crosses between processes once per receiving process set with striping
  (phase 1 carries each message once, phase 2 spreads the stripes inside the set), once per
  receiving process without it ("xferdtensor Transports"; news article, "How NCCL M2N Reshard
  maximizes network bandwidth").
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synthetic as S
from oracle import coracle
from oracle import golden as G

CANARY = 0xA5
POISON = 0x5A


def _one(shape, sm, sp, dm, dp, dtype="bf16"):
    ns, nd = int(np.prod(sm)), int(np.prod(dm))
    t = S.TensorDesc("w", shape, dtype, sm, sp, dm, dp, [S.View(i) for i in range(ns)],
                     [S.View(i) for i in range(nd)], seed=17)
    return S.workloads._size_buffers(S.Workload("one", [t]), ns, nd)


FUZZ = {f"fuzz_{i}": (lambda i=i: S.fuzz_cases(24, seed=29)[i]) for i in range(24)}

WORKLOADS = {
    "dense_tp8_to_dp2tp2": lambda: S.dense_ffn(layers=1, hidden=128, ffn=520),
    "moe_ep4_to_ep2": lambda: S.moe_experts(layers=1, experts=8, hidden=64, ffn=48, ep_src=4, dst="ep2"),
    "replicated_src_to_tp4": lambda: _one((64, 96), (2, 2), ("R", "S0"), (4,), ("S1",)),
    "broadcast_to_4_replicas": lambda: _one((40, 72), (2,), ("S0",), (4,), ("R",), dtype="f32"),
    "transposed_dst": lambda: S.transposed(shape=(96, 80), src_mesh=(2,), src_pl=("S0",), dst_mesh=(2, 2),
                                           dst_pl=("R", "S0")),
    "mesh2x4_to_3x2": lambda: S.mesh2d_to_1d(rows=40, cols=77, variant="2d", dtype="u8"),
    **FUZZ,
}


def owners(wl, layout, world):
    """Process of every flat source and destination pointer index (``random``: seeded draws)."""
    if layout == "random":
        rng = np.random.Generator(np.random.PCG64(len(wl.tensors) * 7919 + world))
        ns, nd = sum(t.n_src for t in wl.tensors), sum(t.n_dst for t in wl.tensors)
        return [int(x) for x in rng.integers(0, world, ns)], [int(x) for x in rng.integers(0, world, nd)]
    so, do = [], []
    for t in wl.tensors:
        for i in range(t.n_src):
            so.append({"colocated": i % world, "disjoint": i % max(1, world // 2),
                       "one_sender": 0}[layout])
        for j in range(t.n_dst):
            do.append({"colocated": j % world, "disjoint": world // 2 + j % (world - world // 2),
                       "one_sender": 1 + j % (world - 1)}[layout])
    return so, do


def table_for(wl, lay, send_n, recv_n):
    es = {k: v[1] for k, v in S.DTYPES.items()}
    src, dst, sc = [], [], []
    for t in wl.tensors:
        for v in t.src_views:
            src.append(("src", lay.src_off[v.buffer], lay.src_off[v.buffer] + wl.src_buffer_numel[v.buffer] * es[t.dtype]))
        for v in t.dst_views:
            dst.append(("dst", lay.dst_off[v.buffer], lay.dst_off[v.buffer] + wl.dst_buffer_numel[v.buffer] * es[t.dtype]))
            sc.append(("none", 0, 0))
    return src + dst + sc + [("send", 0, send_n), ("recv", 0, recv_n)]


def expected_phase1_bytes(R, plan, wl, so, do, striped):
    """Bytes every sender puts on the wire in phase 1, from the method's rule: a region goes once
    to each process set (striped) or once to each process (not striped) holding a destination of
    it other than its sender; the sender is a holder on a receiving process when there is one."""
    total = 0
    regions = R.reshard_plan_regions(plan)
    src_base = np.cumsum([0] + [t.n_src for t in wl.tensors])
    dst_base = np.cumsum([0] + [t.n_dst for t in wl.tensors])
    for i, (ti, s, g, box) in enumerate(regions):
        t = wl.tensors[ti]
        coords = G.mesh_coords(t.src_mesh)
        sbox = G.shard_box(t.global_shape, t.src_mesh, t.src_placements, coords[s])
        holders = [h for h in range(t.n_src)
                   if G.shard_box(t.global_shape, t.src_mesh, t.src_placements, coords[h]) == sbox]
        procs = sorted({do[dst_base[ti] + m] for m in R.reshard_plan_group_members(plan, g)})
        local = [h for h in holders if so[src_base[ti] + h] in procs]
        sender = so[src_base[ti] + (local[0] if local else holders[i % len(holders)])]
        recv = [q for q in procs if q != sender]
        nbytes = int(np.prod([hi - lo for lo, hi in box[:len(t.global_shape)]])) * S.DTYPES[t.dtype][1]
        aligned = (nbytes + 15) // 16 * 16
        if recv:
            total += aligned if striped else aligned * len(recv)
    return total


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, combos, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import dtensor_resharding_gb300 as R
    from dtensor_resharding_gb300 import exchange
    from emulator import run_items
    res = {}
    try:
        for case, layout, striped in combos:
            wl = WORKLOADS[case]()
            lay = S.allocate(wl, "cpu")
            S.fill_sources(wl, lay)
            plan = R.plan_workload(wl)
            so, do = owners(wl, layout, world)
            rp = R.reshard_plan_partition(plan, so, do, world, rank, striped)
            st = R.reshard_plan_stats(rp)
            # this rank's view of memory: other ranks' source buffers poisoned
            src = lay.src_slab.numpy().copy()
            local_src, local_dst = set(), set()
            k = 0
            for t in wl.tensors:
                for v in t.src_views:
                    if so[k] == rank:
                        local_src.add(v.buffer)
                    k += 1
            k = 0
            for t in wl.tensors:
                for v in t.dst_views:
                    if do[k] == rank:
                        local_dst.add(v.buffer)
                    k += 1
            es = {kk: vv[1] for kk, vv in S.DTYPES.items()}
            for b, n in enumerate(wl.src_buffer_numel):
                if b not in local_src:
                    o = lay.src_off[b]
                    src[o: o + n * es[wl.src_buffer_dtype[b]]] = POISON
            send = np.zeros(max(16, st["message_bytes"]), np.uint8)
            recv = np.zeros(max(16, st["recv_bytes"]), np.uint8)
            dst = np.full(lay.dst_slab.numel(), CANARY, np.uint8)
            table = table_for(wl, lay, st["message_bytes"], st["recv_bytes"])
            arrays = {"src": src, "dst": dst, "send": send, "recv": recv}
            run_items(rp, 0, table, arrays, gather=True)   # local copies, gather items included
            run_items(rp, 1, table, arrays)          # outgoing messages
            exchange.run_transfers(rp, torch.from_numpy(send), torch.from_numpy(recv))
            run_items(rp, 2, table, arrays, gather=True)   # received messages
            want = np.full(lay.dst_slab.numel(), CANARY, np.uint8)
            coracle.run_workload(wl, lay.src_slab.numpy(), lay.src_off, want, lay.dst_off)
            bad_local, bad_other = 0, 0
            for b, n in enumerate(wl.dst_buffer_numel):
                o, nb = lay.dst_off[b], n * es[wl.dst_buffer_dtype[b]]
                if b in local_dst:
                    bad_local += int((dst[o: o + nb] != want[o: o + nb]).sum())
                else:
                    bad_other += int((dst[o: o + nb] != CANARY).sum())
            tr = [(p, R.reshard_plan_transfers(rp, p)) for p in (1, 2)]
            res[(case, layout, striped)] = dict(bad_local=bad_local, bad_other=bad_other, stats=st, transfers=tr,
                                                expect1=expected_phase1_bytes(R, plan, wl, so, do, striped))
        out[rank] = res
    finally:
        dist.destroy_process_group()


def _run(world, combos):
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), combos, out), nprocs=world, join=True)
        return dict(out)


def _check(world, res, combos):
    for combo in combos:
        per = [res[r][combo] for r in range(world)]
        for r, x in enumerate(per):
            assert x["bad_local"] == 0, (combo, r, "destination bytes differ from the oracle")
            assert x["bad_other"] == 0, (combo, r, "wrote another rank's destination buffer")
        for phase in (1, 2):
            sends, recvs = {}, {}
            for r, x in enumerate(per):
                for t in dict(x["transfers"])[phase]:
                    key = (r, t["peer"]) if t["dir"] == 0 else (t["peer"], r)
                    (sends if t["dir"] == 0 else recvs).setdefault(key, []).append(t["bytes"])
            assert sends == recvs, (combo, phase, "sends and receives do not pair up")
        sent = sum(x["stats"]["sent_bytes"] for x in per)
        assert sent == per[0]["expect1"], (combo, sent, per[0]["expect1"])
        phase1 = sum(t["bytes"] for x in per for t in dict(x["transfers"])[1] if t["dir"] == 0)
        assert phase1 == sent
        if not combo[2]:
            assert all(x["stats"]["forwarded_bytes"] == 0 for x in per)


COMBOS = [(c, lay, st) for c in sorted(WORKLOADS) if not c.startswith("fuzz") for lay in ("colocated", "disjoint", "one_sender")
          for st in (True, False)]
FUZZ_COMBOS = [(c, "random", i % 2 == 0) for i, c in enumerate(sorted(FUZZ))]


def test_two_gloo_ranks_exchange():
    res = _run(2, COMBOS)
    _check(2, res, COMBOS)


def test_four_gloo_ranks_exchange():
    res = _run(4, COMBOS)
    _check(4, res, COMBOS)
    # striping: the same bytes reach every receiver, but each leaves its sender once
    for c in sorted(w for w in WORKLOADS if not w.startswith("fuzz")):
        for lay in ("colocated", "disjoint", "one_sender"):
            s = sum(res[r][(c, lay, True)]["stats"]["sent_bytes"] for r in range(4))
            f = sum(res[r][(c, lay, True)]["stats"]["forwarded_bytes"] for r in range(4))
            n = sum(res[r][(c, lay, False)]["stats"]["sent_bytes"] for r in range(4))
            assert s + f == n and s <= n
    # a workload with destination replicas on several processes does forward stripes
    assert sum(res[r][("broadcast_to_4_replicas", "one_sender", True)]["stats"]["forwarded_bytes"]
               for r in range(4)) > 0


def test_three_gloo_ranks_fuzzed_layouts_random_owners():
    """Random shapes, meshes, dtypes and per-rank layouts (padded, column-major, offset views)
    with every pointer on a random one of three processes."""
    res = _run(3, FUZZ_COMBOS)
    _check(3, res, FUZZ_COMBOS)


def test_partition_rejects_bad_owners():
    import dtensor_resharding_gb300 as R
    wl = WORKLOADS["dense_tp8_to_dp2tp2"]()
    plan = R.plan_workload(wl)
    so, do = owners(wl, "colocated", 4)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_plan_partition(plan, so, [5] + do[1:], 4, 0)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "dst_owner[0]" in str(e.value)
    with pytest.raises(R.ReshardError):
        R.reshard_plan_partition(plan, so, do, 4, 4)
    rp = R.reshard_plan_partition(plan, so, do, 4, 1)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_plan_partition(rp, so, do, 4, 1)
    assert "already partitioned" in str(e.value)
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute(rp, [1] * plan.n_src_ptrs, [1] * plan.n_dst_ptrs)
    assert "partitioned" in str(e.value)


def test_single_process_partition_is_all_local():
    """With one process every region is a local copy: no messages, no transfers, and the local
    copy table equals the unpartitioned direct table's work."""
    import dtensor_resharding_gb300 as R
    wl = WORKLOADS["dense_tp8_to_dp2tp2"]()
    plan = R.plan_workload(wl)
    rp = R.reshard_plan_partition(plan, [0] * plan.n_src_ptrs, [0] * plan.n_dst_ptrs, 1, 0)
    st, g = R.reshard_plan_stats(rp), R.reshard_plan_stats(plan)
    assert st["message_bytes"] == st["recv_bytes"] == st["transfers"] == 0
    assert st["local_bytes"] == g["bytes_read"] and st["bytes_written"] == g["bytes_written"]


FULL = ["dense_ffn_32x14336x4096_tp8_to_dp2tp2", "moe_8x128x1536x4096_ep16_to_ep8",
        "moe_8x128x1536x4096_ep16_to_tp4_mxfp8", "mesh2x4_to_3x2_14336x4096",
        "transpose_32x14336x4096_tp8_to_dp2tp2_dst_colmajor", "moe_fp8_8x128x768x2048_dp2ep8_to_dp8tp2_b128x128"]


@pytest.mark.parametrize("name", FULL)
def test_partitioned_tables_stay_in_bounds_at_full_size(name):
    """Every item of every pass of every rank's partitioned plan, at full size, reads and writes
    inside its buffers (the send and receive buffers sized by the rank's stats), and the ranks'
    receive buffers together hold every message the senders pack."""
    import dtensor_resharding_gb300 as R
    from test_items_cpu import check_bounds, check_transpose_bounds
    wl = S.workload_by_name(name)
    lay = S.allocate(wl, "meta")
    plan = R.plan_workload(wl)
    quant = wl.quant == "mxfp8"
    for world, layout in ((4, "colocated"), (8, "colocated"), (4, "disjoint")):
        so, do = owners(wl, layout, world)
        sent = recv = 0
        for rank in range(world):
            rp = R.reshard_plan_partition(plan, so, do, world, rank, True)
            st = R.reshard_plan_stats(rp)
            for which in (0, 1, 2):
                check_bounds(wl, lay, rp, which, quant=quant, ws=(st["message_bytes"], st["recv_bytes"]))
                check_transpose_bounds(wl, lay, rp, which, ws=(st["message_bytes"], st["recv_bytes"]))
            ts = R.reshard_plan_transfers(rp, 1) + R.reshard_plan_transfers(rp, 2)
            for t in ts:
                cap = st["message_bytes"] if t["buf"] == R.RESHARD_SEND_BUF else st["recv_bytes"]
                assert t["offset"] % 16 == 0 and t["bytes"] % 16 == 0 and t["offset"] + t["bytes"] <= cap
            sent += sum(t["bytes"] for t in ts if t["dir"] == R.RESHARD_SEND)
            recv += sum(t["bytes"] for t in ts if t["dir"] == R.RESHARD_RECV)
        assert sent == recv


def test_brute_force_partitions_through_the_loopback_transport():
    """120 brute-force problems (every placement kind, nested meshes, uneven and empty chunks,
    element-id payloads), each partitioned over 1-5 processes with random owners, striped or
    not: every rank's emulated pack, the loopback transport and every rank's emulated unpack give
    the oracle's destinations, each rank touching only its own buffers."""
    import dtensor_resharding_gb300 as R
    from dtensor_resharding_gb300 import exchange
    from emulator import run_items
    rng = np.random.Generator(np.random.PCG64(77))
    for i, wl in enumerate(S.brute_force_cases(120, seed=43)):
        world = int(rng.integers(1, 6))
        ns, nd = sum(t.n_src for t in wl.tensors), sum(t.n_dst for t in wl.tensors)
        so = [int(x) for x in rng.integers(0, world, ns)]
        do = [int(x) for x in rng.integers(0, world, nd)]
        lay = S.allocate(wl, "cpu")
        S.fill_sources(wl, lay)
        plan = R.plan_workload(wl)
        want = np.full(lay.dst_slab.numel(), CANARY, np.uint8)
        coracle.run_workload(wl, lay.src_slab.numpy(), lay.src_off, want, lay.dst_off)
        dst = np.full(lay.dst_slab.numel(), CANARY, np.uint8)
        parts, sends, recvs, arrays = [], [], [], []
        for r in range(world):
            rp = R.reshard_plan_partition(plan, so, do, world, r, bool(i % 2))
            st = R.reshard_plan_stats(rp)
            src = lay.src_slab.numpy().copy()
            for k, v in enumerate(wl.tensors[0].src_views):     # one tensor per brute-force case
                if so[k] != r:
                    o = lay.src_off[v.buffer]
                    src[o: o + wl.src_buffer_numel[v.buffer] * S.DTYPES[wl.tensors[0].dtype][1]] = POISON
            send = np.zeros(max(16, st["message_bytes"]), np.uint8)
            recv = np.zeros(max(16, st["recv_bytes"]), np.uint8)
            a = {"src": src, "dst": dst, "send": send, "recv": recv}
            table = table_for(wl, lay, st["message_bytes"], st["recv_bytes"])
            run_items(rp, 0, table, a, gather=True)
            run_items(rp, 1, table, a)
            parts.append((rp, table))
            sends.append(torch.from_numpy(send))
            recvs.append(torch.from_numpy(recv))
            arrays.append(a)
        exchange.loopback_transfers([p for p, _ in parts], sends, recvs)
        for (rp, table), a in zip(parts, arrays):
            run_items(rp, 2, table, a, gather=True)
        assert np.array_equal(dst, want), (i, wl.tensors[0], world, so, do)
