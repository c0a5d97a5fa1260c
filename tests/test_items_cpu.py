"""Device work-item tables checked on the CPU before any kernel runs them.

A host emulation of the device walk (each item: `rows` rows of `run` elements from the source
pointer to every member of its group) applied to host copies of the buffers must reproduce the
oracle byte for byte, and every access of every item (all workloads at full size) must stay
inside the buffer it targets.
"""
import numpy as np
import pytest

import dtensor_resharding_gb300 as R
import synthetic as S
from oracle import coracle

from emulator import run_items
from test_parity_gpu import SMALL

DIRECT, PACK, UNPACK = 0, 1, 2


def _ranges(wl, lay, plan, ws=None):
    """Byte range [lo, hi) in the host slabs of every pointer-table entry (send and receive
    buffers: arrays of their own, `ws` = their sizes; the plan's message bytes by default)."""
    es = {"u8": 1, "bf16": 2, "f16": 2, "f32": 4, "i32": 4, "i64": 8}
    src, dst, sc = [], [], []
    for t in wl.tensors:
        e = es[t.dtype]
        for v in t.src_views:
            src.append(("src", lay.src_off[v.buffer], lay.src_off[v.buffer] + wl.src_buffer_numel[v.buffer] * e))
        for v in t.dst_views:
            de = 1 if wl.quant == "mxfp8" else e
            dst.append(("dst", lay.dst_off[v.buffer], lay.dst_off[v.buffer] + wl.dst_buffer_numel[v.buffer] * de))
            if wl.quant == "mxfp8":
                sc.append(("scale", lay.scale_off[v.buffer], lay.scale_off[v.buffer] + wl.dst_buffer_numel[v.buffer] // 32))
            else:
                sc.append(("none", 0, 0))
    if ws is None:
        n = R.reshard_plan_stats(plan)["message_bytes"]
        ws = (n, n)
    return src + dst + sc + [("ws", 0, ws[0]), ("ws", 0, ws[1])]


def check_bounds(wl, lay, plan, which, quant=False, ws=None):
    items, gs, mp, mo = R.reshard_plan_items(plan, which)
    if len(items) == 0:
        return
    table = _ranges(wl, lay, plan, ws)
    n_dst = plan.n_dst_ptrs
    lo = np.array([r[1] for r in table], np.int64)
    hi = np.array([r[2] for r in table], np.int64)
    es = items["esize"].astype(np.int64)
    src_es = es
    dst_es = np.ones_like(es) if quant and which != PACK else es
    last = (items["rows"].astype(np.int64) - 1)
    s0 = lo[items["src"]] + items["src_off"] * src_es
    s1 = lo[items["src"]] + (items["src_off"] + last * items["src_pitch"] + items["run"]) * src_es
    assert (s0 >= lo[items["src"]]).all() and (s1 <= hi[items["src"]]).all(), "source read out of bounds"
    assert (items["run"] > 0).all() and (items["rows"] > 0).all()
    counts = gs[items["group"] + 1] - gs[items["group"]]
    assert (counts >= 1).all()
    for k in range(int(counts.max())):
        sel = counts > k
        m = gs[items["group"][sel]] + k
        ptr = mp[m]
        off = mo[m]
        it = items[sel]
        d0 = lo[ptr] + (off + it["dst_off"]) * dst_es[sel]
        d1 = lo[ptr] + (off + it["dst_off"] + last[sel] * it["dst_pitch"] + it["run"]) * dst_es[sel]
        assert (d0 >= lo[ptr]).all() and (d1 <= hi[ptr]).all(), "destination write out of bounds"
        if quant and which != PACK:
            e0 = off + it["dst_off"]
            assert (e0 % 32 == 0).all() and (it["run"] % 32 == 0).all() and (it["dst_pitch"] % 32 == 0).all()
            sp = ptr + n_dst
            c1 = lo[sp] + (e0 + last[sel] * it["dst_pitch"] + it["run"]) // 32
            assert (lo[sp] + e0 // 32 >= lo[sp]).all() and (c1 <= hi[sp]).all(), "scale write out of bounds"


def check_transpose_bounds(wl, lay, plan, which, ws=None):
    """Transposing items: every element read and written stays in its buffer, and every item's
    TMA slab coordinates name exactly the element its plain-load offset names, inside a slab that
    lies inside the source buffer."""
    items, gs, mp, mo = R.reshard_plan_items(plan, which + 3)
    if len(items) == 0:
        return
    table = _ranges(wl, lay, plan, ws)
    lo = np.array([r[1] for r in table], np.int64)
    hi = np.array([r[2] for r in table], np.int64)
    es = items["esize"].astype(np.int64)
    rows1 = items["rows"].astype(np.int64) - 1
    cols1 = items["cols"].astype(np.int64) - 1
    s0 = lo[items["src"]] + items["src_off"] * es
    s1 = lo[items["src"]] + (items["src_off"] + rows1 * items["src_pitch"] + cols1 + 1) * es
    assert (s0 >= lo[items["src"]]).all() and (s1 <= hi[items["src"]]).all(), "transpose read out of bounds"
    counts = gs[items["group"] + 1] - gs[items["group"]]
    for k in range(int(counts.max())):
        sel = counts > k
        m = gs[items["group"][sel]] + k
        ptr, off, it = mp[m], mo[m], items[sel]
        d0 = lo[ptr] + (off + it["dst_off"]) * es[sel]
        d1 = lo[ptr] + (off + it["dst_off"] + cols1[sel] * it["dst_pitch"] + rows1[sel] + 1) * es[sel]
        assert (d0 >= lo[ptr]).all() and (d1 <= hi[ptr]).all(), "transpose write out of bounds"
    slabs = np.array(R.reshard_plan_slabs(plan), np.int64).reshape(-1, 6)
    withmap = items[items["slab"] >= 0]
    sl = slabs[withmap["slab"]]
    assert (sl[:, 0] == withmap["src"]).all() and (sl[:, 1] == withmap["esize"]).all()
    assert (sl[:, 2] + withmap["y"] * sl[:, 5] + withmap["x"] == withmap["src_off"]).all()
    assert (withmap["x"] + withmap["cols"] <= sl[:, 3]).all() and (withmap["y"] + withmap["rows"] <= sl[:, 4]).all()
    end = lo[sl[:, 0]] + (sl[:, 2] + (sl[:, 4] - 1) * sl[:, 5] + sl[:, 3]) * sl[:, 1]
    assert (end <= hi[sl[:, 0]]).all(), "a TMA slab reaches past its buffer"


def check_gather_bounds(wl, lay, plan, ws=None, which=None):
    """Pair items of every pass (or of pass `which`): each kind where it belongs (gather rows in
    the direct and unpack passes, scatter rows in the pack pass) with its own invariant, both
    pieces' reads and writes inside their buffers, and a pass's pair items carrying exactly the
    bytes of its copy items flagged as theirs."""
    if which is None:
        for w in (DIRECT, PACK, UNPACK):
            check_gather_bounds(wl, lay, plan, ws, w)
        return
    items, gs, mp, mo = R.reshard_plan_items(plan, 6 + which)
    plain = R.reshard_plan_items(plan, which)[0]
    flagged = plain[plain["pad"][:, 0] == 1]
    assert set(np.unique(plain["pad"][:, 0])) <= {0, 1}
    if len(items) == 0:
        assert len(flagged) == 0
        return
    es = items["esize"].astype(np.int64)
    rows = items["rows"].astype(np.int64)
    assert (rows > 0).all() and (items["run"] >= 2).all()
    if which == PACK:   # one source row into two message blocks
        assert (items["kind"] == 1).all()
        assert (items["src"][:, 1] == items["src"][:, 0]).all()
        assert (items["src_off"][:, 1] == items["src_off"][:, 0] + items["run"][:, 0]).all()
    else:               # one destination row of two pieces side by side
        assert (items["kind"] == 0).all()
        assert (items["dst_off"][:, 1] == items["dst_off"][:, 0] + items["run"][:, 0]).all()
        assert (items["dst_pitch"][:, 1] == items["dst_pitch"][:, 0]).all()
    assert int((rows * (items["run"][:, 0] + items["run"][:, 1]) * es).sum()) == \
        int((flagged["rows"].astype(np.int64) * flagged["run"] * flagged["esize"]).sum())
    table = _ranges(wl, lay, plan, ws)
    lo = np.array([r[1] for r in table], np.int64)
    hi = np.array([r[2] for r in table], np.int64)
    counts = gs[items["group"] + 1] - gs[items["group"]]
    for p in (0, 1):
        sp = items["src"][:, p]
        s0 = lo[sp] + items["src_off"][:, p] * es
        s1 = lo[sp] + (items["src_off"][:, p] + (rows - 1) * items["src_pitch"][:, p] + items["run"][:, p]) * es
        assert (s0 >= lo[sp]).all() and (s1 <= hi[sp]).all(), "pair item read out of bounds"
        for k in range(int(counts.max())):
            sel = counts > k
            m = gs[items["group"][sel]] + k
            ptr, off, it = mp[m], mo[m], items[sel]
            d0 = lo[ptr] + (off + it["dst_off"][:, p]) * es[sel]
            d1 = lo[ptr] + (off + it["dst_off"][:, p] + (rows[sel] - 1) * it["dst_pitch"][:, p] + it["run"][:, p]) * es[sel]
            assert (d0 >= lo[ptr]).all() and (d1 <= hi[ptr]).all(), "pair item write out of bounds"


def emulate(wl, lay, plan, mode, gather=False):
    """Apply the item tables to host copies of the slabs (plain copies only); with `gather`, the
    direct pass as the executor runs it when the plan has gather items."""
    src = lay.src_slab.numpy()
    dst = np.full(lay.dst_slab.numel(), 0xA5, np.uint8)
    ws = np.zeros(max(1, R.reshard_plan_stats(plan)["message_bytes"]), np.uint8)
    table = _ranges(wl, lay, plan)
    arrays = {"src": src, "dst": dst, "ws": ws}
    for which in ((DIRECT,) if mode == "direct" else (PACK, UNPACK)):
        run_items(plan, which, table, arrays, gather=gather)
    return dst


def _oracle(wl, lay):
    want = np.full(lay.dst_slab.numel(), 0xA5, np.uint8)
    coracle.run_workload(wl, lay.src_slab.numpy(), lay.src_off, want, lay.dst_off)
    return want


@pytest.mark.parametrize("mode", ["direct", "packed"])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_item_tables_reproduce_oracle(name, mode):
    wl = SMALL[name]()
    lay = S.allocate(wl, "cpu", misalign=2 if all(t.dtype in ("bf16", "u8") for t in wl.tensors) else 0)
    S.fill_sources(wl, lay)
    plan = R.plan_workload(wl)
    for which in (DIRECT, PACK, UNPACK):
        check_bounds(wl, lay, plan, which)
        check_transpose_bounds(wl, lay, plan, which)
    check_gather_bounds(wl, lay, plan)
    want = _oracle(wl, lay)
    assert np.array_equal(emulate(wl, lay, plan, mode), want)
    assert np.array_equal(emulate(wl, lay, plan, mode, gather=True), want)


def test_item_tables_brute_force():
    for wl in S.brute_force_cases(120, seed=41):
        lay = S.allocate(wl, "cpu")
        S.fill_sources(wl, lay)
        plan = R.plan_workload(wl)
        for which in (DIRECT, PACK, UNPACK):
            check_bounds(wl, lay, plan, which)
        check_gather_bounds(wl, lay, plan)
        want = _oracle(wl, lay)
        for mode in ("direct", "packed"):
            assert np.array_equal(emulate(wl, lay, plan, mode), want)
            assert np.array_equal(emulate(wl, lay, plan, mode, gather=True), want)


@pytest.mark.parametrize("case", ["moe_tp4", "six_replicas"])
def test_mxfp8_item_tables_small(case):
    if case == "moe_tp4":
        wl = S.moe_experts(layers=1, experts=16, hidden=256, ffn=256, dst="tp4")
    else:  # more destination replicas than one quantizer pass writes
        from test_parity_gpu import _one
        wl = _one((64, 128), (2,), ("S0",), (6, 2), ("R", "S1"), quant="mxfp8")
    lay = S.allocate(wl, "meta")
    plan = R.plan_workload(wl)
    # the plan accepts MXFP8: with NULL pointers the execute stops at the pointer check
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute(plan, [0] * plan.n_src_ptrs, [0] * (2 * plan.n_dst_ptrs), quant="mxfp8")
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG
    for which in (DIRECT, PACK, UNPACK):
        check_bounds(wl, lay, plan, which, quant=True)


@pytest.mark.parametrize("name", sorted(S.WORKLOAD_NAMES))
def test_full_size_item_bounds(name):
    """Every item of every pass of every full-size workload stays inside its buffers."""
    wl = S.workload_by_name(name)
    lay = S.allocate(wl, "meta")
    plan = R.plan_workload(wl)
    for which in (DIRECT, PACK, UNPACK):
        check_bounds(wl, lay, plan, which, quant=wl.quant == "mxfp8")
        check_transpose_bounds(wl, lay, plan, which)
    check_gather_bounds(wl, lay, plan)


# rows of a misaligned column split assembled from two source pieces, as (piece 0, piece 1)
# bytes: 1024-column source shards of a 2 x 4 mesh into destinations of 1366, 1366 and 1364
# columns (torch.chunk of 4096 by 3)
MESH_PIECES = {(2048, 684), (1364, 1368), (680, 2048)}
GATHER_EXPECT = {name: MESH_PIECES for name in ("mesh2x4_to_3_14336x4096", "mesh2x4_to_3x2_14336x4096",
                                                "mesh2x4_to_3_57344x4096", "mesh2x4_to_3x2_57344x4096")}


@pytest.mark.parametrize("name", sorted(S.WORKLOAD_NAMES))
def test_gather_items_where_rows_are_split_and_misaligned(name):
    """Gather items appear exactly where a destination row is two source pieces and the rows are
    misaligned by construction; their pieces are the expected column splits, every row of every
    paired region is covered, and a region is paired at most once."""
    wl = S.workload_by_name(name)
    plan = R.plan_workload(wl)
    items = R.reshard_plan_items(plan, 6)[0]
    unpack = R.reshard_plan_items(plan, 8)[0]
    pack = R.reshard_plan_items(plan, 7)[0]
    assert R.reshard_plan_stats(plan)["gather_items"] == len(items) + len(pack) + len(unpack)
    if name not in GATHER_EXPECT:
        assert len(items) == 0 and len(unpack) == 0, name
        return
    # the pack pass splits each source row that feeds two destinations (the (2,4) source's
    # 1024-column shards 1 and 2: 684 + 1364 and 1368 + 680 bytes) into its two message blocks
    es_p = pack["esize"].astype(np.int64)
    assert {(int(a), int(b)) for a, b in zip(pack["run"][:, 0] * es_p, pack["run"][:, 1] * es_p)} == \
        {(684, 1364), (1368, 680)}
    # the unpack pass pairs the same rows (pieces read from the received message)
    es = unpack["esize"].astype(np.int64)
    assert {(int(a), int(b)) for a, b in zip(unpack["run"][:, 0] * es, unpack["run"][:, 1] * es)} == GATHER_EXPECT[name]
    assert int(unpack["rows"].sum()) == int(items["rows"].sum())
    es = items["esize"].astype(np.int64)
    got = {(int(a), int(b)) for a, b in zip(items["run"][:, 0] * es, items["run"][:, 1] * es)}
    assert got == GATHER_EXPECT[name]
    assert (items["dst_pitch"][:, 0] * es == (items["run"][:, 0] + items["run"][:, 1]) * es).all()
    t = wl.tensors[0]
    n_rep = int(np.prod(t.dst_mesh)) // 3
    gs = R.reshard_plan_items(plan, 6)[1]
    assert all(gs[g + 1] - gs[g] == n_rep for g in items["group"])
    # every destination row of the tensor is written by exactly one gather item
    assert int(items["rows"].sum()) == t.global_shape[0] * 3


def test_gather_pairs_follow_the_alignment_rule():
    """A column split whose pieces and destination pitch are 16-byte multiples pairs nothing;
    one whose destination pitch is not pairs every row; a replicated source counts once."""
    from test_parity_gpu import _one
    aligned = _one((64, 1024), (2,), ("S1",), (4,), ("S1",))           # 512-col pieces, 256-col rows
    assert R.reshard_plan_stats(R.plan_workload(aligned))["gather_items"] == 0
    split = _one((64, 1000), (4,), ("S1",), (3,), ("S1",))             # 250-col sources, 334-col rows
    st = R.reshard_plan_stats(R.plan_workload(split))
    assert st["gather_items"] > 0
    items = R.reshard_plan_items(R.plan_workload(split), 6)[0]
    assert int(items["rows"].sum()) == 64 * 3
    rep = _one((64, 1000), (2, 4), ("R", "S1"), (3,), ("S1",))         # the same with two replicas
    items2 = R.reshard_plan_items(R.plan_workload(rep), 6)[0]
    assert int(items2["rows"].sum()) == 64 * 3


@pytest.mark.parametrize("ns,nd,per_row", [(8, 2, 4), (9, 3, 3)])
def test_gather_pairs_rows_of_more_pieces(ns, nd, per_row):
    """Rows of four pieces form two gather pairs; rows of three form one pair and keep the last
    piece as a plain item. Both emulate to the oracle."""
    from test_parity_gpu import _split
    wl = _split((64, ns * 111), ns, nd)
    plan = R.plan_workload(wl)
    items = R.reshard_plan_items(plan, 6)[0]
    plain = R.reshard_plan_items(plan, DIRECT)[0]
    pairs = per_row // 2
    assert int(items["rows"].sum()) == 64 * nd * pairs
    unflagged = plain[plain["pad"][:, 0] == 0]
    assert int((unflagged["rows"].astype(np.int64) * unflagged["run"]).sum()) == 64 * nd * (per_row % 2) * 111
    lay = S.allocate(wl, "cpu", misalign=2)
    S.fill_sources(wl, lay)
    check_gather_bounds(wl, lay, plan)
    for mode in ("direct", "packed"):
        assert np.array_equal(emulate(wl, lay, plan, mode, gather=True), _oracle(wl, lay))


def test_gather_items_merge_outer_dims():
    """A 3-D column split whose middle dim is short: outer dims merge into the gather items' rows
    when both sources and the destination step uniformly over them (64 x 3 rows per pair, not 64
    items of 3 rows), and the tables still reproduce the oracle; a padded destination pitch on
    the outer dim keeps them apart."""
    from test_parity_gpu import _split
    wl = _split((64, 3, 1000), 4, 3)
    plan = R.plan_workload(wl)
    items = R.reshard_plan_items(plan, 6)[0]
    assert int(items["rows"].sum()) == 64 * 3 * 3
    assert len(items) <= 3 * -(-64 * 3 // 8)
    unpack = R.reshard_plan_items(plan, 8)[0]   # message blocks are dense: their rows merge too
    assert int(unpack["rows"].sum()) == 64 * 3 * 3 and len(unpack) == len(items)
    lay = S.allocate(wl, "cpu", misalign=2)
    S.fill_sources(wl, lay)
    check_gather_bounds(wl, lay, plan)
    assert np.array_equal(emulate(wl, lay, plan, "direct", gather=True), _oracle(wl, lay))
    assert np.array_equal(emulate(wl, lay, plan, "packed", gather=True), _oracle(wl, lay))
    # destination shards with a padded outer stride: the outer dim is walked explicitly
    t = wl.tensors[0]
    cols = [334, 334, 332]   # torch.chunk of 1000 columns into 3
    t.dst_views = [S.View(i, 0, (3 * c + 8, c, 1)) for i, c in enumerate(cols)]
    wl = S.workloads._size_buffers(S.Workload("padded", [t]), 4, 3)
    plan = R.plan_workload(wl)
    items = R.reshard_plan_items(plan, 6)[0]
    assert len(items) == 3 * 64 and (items["rows"] == 3).all()
    lay = S.allocate(wl, "cpu")
    S.fill_sources(wl, lay)
    check_gather_bounds(wl, lay, plan)
    assert np.array_equal(emulate(wl, lay, plan, "direct", gather=True), _oracle(wl, lay))


def test_item_tables_fuzzed_layouts():
    """Random shapes, meshes, dtypes and per-rank layouts (dense, padded, column-major, offset)."""
    for wl in S.fuzz_cases(60, seed=23):
        lay = S.allocate(wl, "cpu")
        S.fill_sources(wl, lay)
        plan = R.plan_workload(wl)
        for which in (DIRECT, PACK, UNPACK):
            check_bounds(wl, lay, plan, which)
            check_transpose_bounds(wl, lay, plan, which)
        check_gather_bounds(wl, lay, plan)
        want = _oracle(wl, lay)
        for mode in ("direct", "packed"):
            assert np.array_equal(emulate(wl, lay, plan, mode), want), (wl.tensors[0], mode)
            assert np.array_equal(emulate(wl, lay, plan, mode, gather=True), want), (wl.tensors[0], mode)
