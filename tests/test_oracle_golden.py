"""Pins for the golden reshard oracle (CPU only).

Each check is written as a function of the oracle pieces it pins, so that the mutation tests
can feed it a deliberately broken oracle and see it fail.
"""
import itertools

import numpy as np
import pytest
import torch

import synthetic as S
from oracle import golden as G
from oracle import coracle as C

from conftest import read_fixture


# ------------------------------------------------------------------ chunk rule: torch.chunk

def check_chunk_rule(chunk_bounds):
    """torch.chunk is the library definition of a DTensor Shard split (uneven, empty tail)."""
    for length in range(0, 41):
        for n in range(1, 10):
            parts = torch.chunk(torch.arange(length), n) if length else ()
            for i in range(n):
                lo, hi = chunk_bounds(length, n, i)
                if i < len(parts) and length:
                    p = parts[i]
                    assert (lo, hi) == (int(p[0]), int(p[-1]) + 1), (length, n, i)
                else:
                    assert hi - lo == 0, (length, n, i)


def test_chunk_rule_matches_torch_chunk():
    check_chunk_rule(G.chunk_bounds)


def test_chunk_rule_printed_sizes():
    # 14336 rows over TP6: five chunks of 2390 and one of 2386; over TP5: four of 2868, one of
    # 2864; 4096 columns over 3: 1366, 1366, 1364 (closed form ceil(L/n)).
    assert [G.chunk_bounds(14336, 6, i)[1] - G.chunk_bounds(14336, 6, i)[0] for i in range(6)] == [2390] * 5 + [2386]
    assert [G.chunk_bounds(14336, 5, i)[1] - G.chunk_bounds(14336, 5, i)[0] for i in range(5)] == [2868] * 4 + [2864]
    assert [G.chunk_bounds(4096, 3, i)[1] - G.chunk_bounds(4096, 3, i)[0] for i in range(3)] == [1366, 1366, 1364]
    assert [G.chunk_bounds(5, 4, i) for i in range(4)] == [(0, 2), (2, 4), (4, 5), (5, 5)]


def check_nested_boxes(shard_box):
    """Boxes equal the ids that nested torch.chunk leaves each rank (brute-force meshes)."""
    rng = np.random.Generator(np.random.PCG64(11))
    for _ in range(300):
        nd = int(rng.integers(1, 4))
        shape = tuple(int(x) for x in rng.integers(1, 10, size=nd))
        md = int(rng.integers(1, 4))
        mesh = tuple(int(x) for x in rng.integers(1, 5, size=md))
        pls = tuple("R" if c == nd else f"S{c}" for c in rng.integers(0, nd + 1, size=md))
        ids = torch.arange(int(np.prod(shape))).reshape(shape)
        for coord in itertools.product(*[range(m) for m in mesh]):
            want = S.workloads._chunk_local(ids, mesh, pls, coord)
            box = shard_box(shape, mesh, pls, coord)
            got = ids[tuple(slice(lo, hi) for lo, hi in box)]
            assert tuple(got.shape) == tuple(want.shape), (shape, mesh, pls, coord)
            assert torch.equal(got, want), (shape, mesh, pls, coord)


def test_nested_boxes_match_torch_chunk():
    check_nested_boxes(G.shard_box)


# ------------------------------------------------------------------ the 8x8 worked example

def check_example_8x8(source_regions, golden_reshard):
    rows, _ = read_fixture("example_8x8.txt")
    want = sorted(((int(d),), int(s), ((int(r0), int(r1)), (int(c0), int(c1))))
                  for d, s, r0, r1, c0, c1 in rows)
    wl = S.example_8x8()
    desc = wl.tensors[0]
    assert source_regions(desc) == want
    # values: source r holds rows 4r..4r+3 of M; destination j must hold columns 2j, 2j+1
    m = np.arange(64, dtype=np.int32).reshape(8, 8)
    d = S.TensorDesc("m", (8, 8), "i32", (2,), ("S0",), (4,), ("S1",),
                     [S.View(0), S.View(1)], [S.View(i) for i in range(4)])
    src = [m[4 * r: 4 * r + 4].copy().view(np.uint8).reshape(-1) for r in range(2)]
    dst = [np.zeros(8 * 2 * 4, np.uint8) for _ in range(4)]
    golden_reshard(d, src, dst)
    for j in range(4):
        assert np.array_equal(dst[j].view(np.int32).reshape(8, 2), m[:, 2 * j: 2 * j + 2])
    # eight 4x2 regions, 128 bytes of bf16 moved in total
    assert len(want) == 8
    assert sum((r1 - r0) * (c1 - c0) * 2 for _, _, ((r0, r1), (c0, c1)) in want) == 128


def test_example_8x8():
    check_example_8x8(G.source_regions, G.golden_reshard)


def test_tp4_to_tp2dp2_replica_example():
    rows, meta = read_fixture("tp4_to_tp2dp2.txt")
    want = sorted((tuple(int(x) for x in g.split(",")), int(s), ((int(r0), int(r1)), (int(c0), int(c1))))
                  for g, s, r0, r1, c0, c1 in rows)
    d = S.TensorDesc("w", (8, 4), "i32", (4,), ("S0",), (2, 2), ("R", "S0"),
                     [S.View(i) for i in range(4)], [S.View(i) for i in range(4)])
    assert G.source_regions(d) == want
    acc = G.byte_accounting(d)
    assert acc["bytes_read"] == int(meta["bytes_read"][0])
    assert acc["bytes_written"] == int(meta["bytes_written"][0])
    assert acc["gather_bcast_bytes"] == 2 * 8 * 4 * 4


# ------------------------------------------------------------------ brute force coverage

def _run_oracle(wl, impl="py"):
    lay = S.allocate(wl, "cpu")
    S.fill_sources(wl, lay)
    S.fill_canary(lay)
    src = lay.src_slab.numpy()
    dst = lay.dst_slab.numpy().copy()
    sc = lay.scale_slab.numpy().copy() if lay.scale_slab is not None else None
    mod = G if impl == "py" else C
    mod.run_workload(wl, src, lay.src_off, dst, lay.dst_off, sc, lay.scale_off)
    return lay, dst, sc


def check_brute_force(run):
    """Every destination element carries its own global id (element-id payload)."""
    for wl in S.brute_force_cases(150, seed=5):
        t = wl.tensors[0]
        lay, dst, _ = run(wl)
        ids = torch.arange(int(np.prod(t.global_shape)), dtype=torch.int32).reshape(t.global_shape)
        for coord, v in zip(itertools.product(*[range(m) for m in t.dst_mesh]), t.dst_views):
            want = S.workloads._chunk_local(ids, t.dst_mesh, t.dst_placements, coord).contiguous().numpy()
            off = lay.dst_off[v.buffer]
            got = dst[off: off + want.size * 4].view(np.int32).reshape(want.shape)
            assert np.array_equal(got, want), (t.global_shape, t.src_mesh, t.src_placements,
                                               t.dst_mesh, t.dst_placements, coord)


def test_brute_force_python_oracle():
    check_brute_force(lambda wl: _run_oracle(wl, "py"))


def test_brute_force_c_oracle():
    check_brute_force(lambda wl: _run_oracle(wl, "c"))


def test_uncovered_and_replica_mismatch_detected():
    d = S.TensorDesc("w", (4, 4), "i32", (2,), ("R",), (2,), ("S0",),
                     [S.View(0), S.View(1)], [S.View(0), S.View(1)])
    a = np.arange(16, dtype=np.int32).view(np.uint8)
    b = a.copy()
    b[4] ^= 1
    with pytest.raises(G.OracleError):
        G.golden_reshard(d, [a, b], [np.zeros(32, np.uint8)] * 2)
    with pytest.raises(RuntimeError):
        C.reshard_tensor(d, [a, b], [np.zeros(32, np.uint8), np.zeros(32, np.uint8)])


# ------------------------------------------------------------------ invariants

def test_round_trip_identity():
    """A -> B -> A reproduces the source buffers byte for byte (zero changed parameters)."""
    for wl in S.brute_force_cases(60, seed=9):
        t = wl.tensors[0]
        lay, dst, _ = _run_oracle(wl)
        back = S.TensorDesc("back", t.global_shape, t.dtype, t.dst_mesh, t.dst_placements,
                            t.src_mesh, t.src_placements, t.dst_views, t.src_views)
        es = G.ESIZE[t.dtype]
        src_np = lay.src_slab.numpy()
        sb = [dst[lay.dst_off[v.buffer]: lay.dst_off[v.buffer] + wl.dst_buffer_numel[v.buffer] * es]
              for v in back.src_views]
        out = [np.full(wl.src_buffer_numel[v.buffer] * es, 0xA5, np.uint8) for v in back.dst_views]
        G.golden_reshard(back, sb, out)
        for v, o in zip(t.src_views, out):
            ref = src_np[lay.src_off[v.buffer]: lay.src_off[v.buffer] + wl.src_buffer_numel[v.buffer] * es]
            assert np.array_equal(o, ref)


def test_byte_accounting_closed_forms():
    # dense FFN at small size: written = DP x S, read = S, gather+bcast = 2 S
    wl = S.dense_ffn(layers=1, hidden=64, ffn=96)
    for t in wl.tensors:
        acc = G.byte_accounting(t)
        total = int(np.prod(t.global_shape)) * 2
        assert acc["bytes_read"] == total
        assert acc["bytes_written"] == 2 * total
        assert acc["gather_bcast_bytes"] == 2 * total
        assert acc["dst_groups"] == 2


def test_fused_gate_up_views_c_vs_python():
    for fused in ("block", "interleave", "none"):
        wl = S.dense_ffn(layers=2, hidden=48, ffn=200, tp_src=8, fused=fused)
        _, d_py, _ = _run_oracle(wl, "py")
        _, d_c, _ = _run_oracle(wl, "c")
        assert np.array_equal(d_py, d_c)


def test_uneven_and_2d_mesh_c_vs_python():
    for wl in (S.uneven_tp(rows=143, cols=40, src=6, dst=5), S.mesh2d_to_1d(rows=30, cols=41, variant="1d"),
               S.mesh2d_to_1d(rows=30, cols=41, variant="2d"), S.many_small(n=12, rows=(1, 20), cols=(1, 9))):
        _, d_py, _ = _run_oracle(wl, "py")
        _, d_c, _ = _run_oracle(wl, "c")
        assert np.array_equal(d_py, d_c), wl.name


def test_dst_element_source_matches_golden():
    wl = S.mesh2d_to_1d(rows=30, cols=41, variant="2d")
    lay, dst, _ = _run_oracle(wl)
    t = wl.tensors[0]
    src = lay.src_slab.numpy()
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(200):
        r = int(rng.integers(0, t.n_dst))
        coord = G.mesh_coords(t.dst_mesh)[r]
        shp = G.box_shape(G.shard_box(t.global_shape, t.dst_mesh, t.dst_placements, coord))
        idx = tuple(int(rng.integers(0, n)) for n in shp)
        s, sidx = G.dst_element_source(t, r, idx)
        sshp = G.box_shape(G.shard_box(t.global_shape, t.src_mesh, t.src_placements, G.mesh_coords(t.src_mesh)[s]))
        so = lay.src_off[t.src_views[s].buffer] + 2 * G.element_offset(t.src_views[s], sshp, sidx)
        do = lay.dst_off[t.dst_views[r].buffer] + 2 * G.element_offset(t.dst_views[r], shp, idx)
        assert bytes(src[so:so + 2]) == bytes(dst[do:do + 2])
