"""Pins for the oracle's whole-reshard MXFP8 branch (CPU only): where codes and scales land.

The element rule is pinned elsewhere (brute force over every BF16 pattern). Here the reshard
branches that place a quantized shard are pinned:
- a hand-derived fixture (tests/golden/mxfp8_placement_2x128.txt) lists every scale byte and
  every block of codes of a tiny reshard whose values make each block's scale and second code
  name the block, with two shards in one buffer at offsets 0 and 160;
- the C oracle and the Python oracle, written independently, agree byte for byte (codes and
  scales) on MoE expert tensors split for TP4, a six-way replicated destination, shards at
  offsets inside shared buffers, 3-D tensors, zero blocks and Inf/NaN blocks;
- planted mistakes in either oracle's placement (scale base at the element offset instead of
  offset / 32, a scale row stride of K instead of K / 32, codes of a block at the wrong byte)
  fail the fixture.
"""
import os
import subprocess

import numpy as np
import pytest

import synthetic as S
from oracle import coracle as C
from oracle import golden as G

from conftest import read_fixture

FIX = "mxfp8_placement_2x128.txt"
CANARY = 0xA5


def _bf16_pow2(k: int, negative: bool = False) -> int:
    return (0x8000 if negative else 0) | ((k + 127) << 7)


def fixture_values() -> np.ndarray:
    """The fixture's [2, 128] BF16 bit patterns, from its value rule."""
    v = np.zeros((2, 128), np.uint16)
    for row in range(2):
        for col in range(128):
            g, j = 4 * row + col // 32, col % 32
            if j == 0:
                b = _bf16_pow2(g - 3)
            elif j == 1:
                b = ((g - 4 + 127) << 7) | (16 * g)     # (1 + g/8) * 2^(g-4)
            elif j % 2:
                b = _bf16_pow2(g - 4, negative=True)
            else:
                b = _bf16_pow2(g - 5)
            v[row, col] = b
    return v


def fixture_workload():
    rows, meta = read_fixture(FIX)
    offs = [int(x) for x in meta["dst_offsets"]]
    t = S.TensorDesc("w", (2, 128), "bf16", (1,), ("R",), (2,), ("S1",), [S.View(0)],
                     [S.View(0, offs[0]), S.View(0, offs[1])])
    wl = S.Workload("mxfp8_placement", [t], quant="mxfp8",
                    src_buffer_numel=[256], src_buffer_dtype=["bf16"],
                    dst_buffer_numel=[int(meta["data_bytes"][0])], dst_buffer_dtype=["u8"])
    return wl, rows


def expected_from_fixture(rows, n_data, n_scale):
    data = np.full(n_data, CANARY, np.uint8)
    scale = np.full(n_scale, CANARY, np.uint8)
    for r in rows:
        if r[0] == "scale":
            scale[int(r[1])] = int(r[2])
        elif r[0] == "block":
            first, g = int(r[1]), int(r[2])
            blk = [0x78, 0x70 | g] + [0xF0 if j % 2 else 0x68 for j in range(2, 32)]
            data[first: first + 32] = blk
    return data, scale


def run_fixture(runner):
    """Run one oracle on the fixture problem. The scale buffer is as long as the data buffer so
    that a planted mistake that writes past the 9 scale bytes stays inside it (and is seen)."""
    wl, rows = fixture_workload()
    src = fixture_values().reshape(-1).view(np.uint8).copy()
    n = wl.dst_buffer_numel[0]
    data = np.full(n, CANARY, np.uint8)
    scale = np.full(n, CANARY, np.uint8)
    runner(wl, src, [0], data, [0], scale, [0])
    return wl, rows, data, scale


def check_fixture(runner):
    wl, rows, data, scale = run_fixture(runner)
    want_d, want_s = expected_from_fixture(rows, data.size, scale.size)
    bad = np.nonzero(data != want_d)[0]
    assert bad.size == 0, f"{bad.size} data bytes differ from the fixture, first at {bad[:6]}"
    bad = np.nonzero(scale != want_s)[0]
    assert bad.size == 0, f"{bad.size} scale bytes differ from the fixture, first at {bad[:6]}"


def test_fixture_value_rule_is_what_it_says():
    """The constructed values are the fixture's: amax 2^(g-3) at j = 0, and so on."""
    v = fixture_values().astype(np.uint32) << 16
    f = v.view(np.float32).astype(np.float64)
    for row in range(2):
        for b in range(4):
            g = 4 * row + b
            blk = f[row, 32 * b: 32 * b + 32]
            assert np.abs(blk).max() == 2.0 ** (g - 3)
            assert blk[1] == (1 + g / 8) * 2.0 ** (g - 4)


def test_c_oracle_matches_hand_derived_placement():
    check_fixture(lambda *a: C.run_workload(*a))


def test_python_oracle_matches_hand_derived_placement():
    check_fixture(lambda *a: G.run_workload(*a))


# ----------------------------------------------------------------- the two oracles agree

def _one(shape, sm, sp, dm, dp, dst_views=None, dst_numel=None, seed=31):
    ns, nd = int(np.prod(sm)), int(np.prod(dm))
    dv = dst_views or [S.View(i) for i in range(nd)]
    t = S.TensorDesc("w", shape, "bf16", sm, sp, dm, dp, [S.View(i) for i in range(ns)], dv, seed=seed)
    wl = S.workloads._size_buffers(S.Workload("one", [t], quant="mxfp8"), ns, max(v.buffer for v in dv) + 1)
    if dst_numel:
        wl.dst_buffer_numel = list(dst_numel)
    return wl


def _shared_buffer_case():
    """Two tensors whose destination shards share buffers at offsets (multiples of 32)."""
    a = S.TensorDesc("a", (3, 10, 96), "bf16", (2,), ("S1",), (2,), ("S0",), [S.View(0), S.View(1)],
                     [S.View(0, 0), S.View(0, 2 * 10 * 96 + 96)], seed=41)
    b = S.TensorDesc("b", (40, 64), "bf16", (4,), ("S0",), (2, 2), ("R", "S1"),
                     [S.View(2 + i) for i in range(4)],
                     [S.View(1, 0), S.View(1, 40 * 32 + 64), S.View(2, 32), S.View(2, 32 + 40 * 32 + 64)], seed=42)
    return S.workloads._size_buffers(S.Workload("shared_buffers", [a, b], quant="mxfp8"), 6, 3)


CASES = {
    "moe_tp4": lambda: S.moe_experts(layers=1, experts=4, hidden=64, ffn=128, ep_src=2, dst="tp4"),
    "six_replicas": lambda: _one((64, 128), (2,), ("S0",), (6, 2), ("R", "S1")),
    "shards_at_offsets_in_shared_buffers": _shared_buffer_case,
    "uneven_rows_3d": lambda: _one((5, 7, 64), (3,), ("S1",), (2,), ("S0",)),
}


def _host_layout(wl, specials=False):
    lay = S.allocate(wl, "cpu", misalign=0)
    S.fill_sources(wl, lay)
    src = lay.src_slab.numpy()
    if specials:
        # zero blocks, a -0 block, Inf and NaN blocks, subnormals (sources are disjoint here)
        u16 = src.view(np.uint16)
        rng = np.random.Generator(np.random.PCG64(3))
        pats = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC1, 0x0001, 0x8001, 0x007F, 0x43E0, 0x43F0,
                         0x4400, 0x3F88, 0xBF88, 0x7F7F, 0xFF7F, 0x3A80], np.uint16)
        pick = rng.random(u16.size) < 0.05
        u16[pick] = pats[rng.integers(0, pats.size, pick.sum())]
        nb = u16.size // 32
        for k in rng.integers(0, nb, 8):
            u16[32 * k: 32 * k + 32] = 0
        for k in rng.integers(0, nb, 4):
            u16[32 * k: 32 * k + 32] = 0x8000
    return lay, src


def _both(wl, lay, src):
    out = []
    for run in (C.run_workload, G.run_workload):
        data = np.full(lay.dst_slab.numel(), CANARY, np.uint8)
        scale = np.full(lay.scale_slab.numel(), CANARY, np.uint8)
        run(wl, src, lay.src_off, data, lay.dst_off, scale, lay.scale_off)
        out.append((data, scale))
    return out


@pytest.mark.parametrize("name", sorted(CASES))
def test_c_and_python_mxfp8_reshards_agree(name):
    wl = CASES[name]()
    lay, src = _host_layout(wl)
    (cd, cs), (pd, ps) = _both(wl, lay, src)
    assert np.array_equal(cd, pd), f"{name}: codes differ at {np.nonzero(cd != pd)[0][:8]}"
    assert np.array_equal(cs, ps), f"{name}: scales differ at {np.nonzero(cs != ps)[0][:8]}"
    # every byte inside a view was written: the canary survives only outside the views
    written = int((cd != CANARY).sum())
    n_el = sum(int(np.prod(G.box_shape(G.shard_box(t.global_shape, t.dst_mesh, t.dst_placements, c))))
               for t in wl.tensors for c in G.mesh_coords(t.dst_mesh))
    assert written > 0.95 * n_el


def test_c_and_python_agree_on_special_blocks():
    wl = CASES["moe_tp4"]()
    lay, src = _host_layout(wl, specials=True)
    (cd, cs), (pd, ps) = _both(wl, lay, src)
    assert np.array_equal(cd, pd) and np.array_equal(cs, ps)
    assert (cs == 0xFF).any() and (cs == 0x00).any()     # NaN scales and zero-block scales occur


# ------------------------------------------------------------------------ planted mistakes

def _mutant_c(tmp_path, old, new):
    """A build of oracle.c with one planted mistake (text replaced), loaded beside the real one."""
    src = open(os.path.join(os.path.dirname(C.__file__), "oracle.c")).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", str(path), "-o", str(so)], check=True)
    return C.load(str(so))


C_MUTANTS = {
    "scale_base_is_the_element_offset": ("d_scales[r] + d_off[r] / 32 + row * nb + b",
                                         "d_scales[r] + d_off[r] + row * nb + b"),
    "scale_row_stride_is_K": ("d_scales[r] + d_off[r] / 32 + row * nb + b",
                              "d_scales[r] + d_off[r] / 32 + row * ext[nd - 1] + b"),
    "codes_of_a_block_one_byte_per_block": ("d_bufs[r] + l0 + 32 * b,", "d_bufs[r] + l0 + b,"),
}


@pytest.mark.parametrize("mutant", sorted(C_MUTANTS))
def test_planted_mistakes_in_the_c_oracle_are_caught(mutant, tmp_path):
    L = _mutant_c(tmp_path, *C_MUTANTS[mutant])
    with pytest.raises(AssertionError):
        check_fixture(lambda *a: C.run_workload(*a, L=L))


def _scale_base_at_offset(data_buf, scale_buf, offset, codes, scales):
    c = np.asarray(codes, np.uint8).reshape(-1)
    s = np.asarray(scales, np.uint8).reshape(-1)
    data_buf[offset: offset + c.size] = c
    scale_buf[offset: offset + s.size] = s


def _scale_stride_k(data_buf, scale_buf, offset, codes, scales):
    c = np.asarray(codes, np.uint8).reshape(-1)
    data_buf[offset: offset + c.size] = c
    k = len(codes[0])
    for r, row in enumerate(scales):
        scale_buf[offset // 32 + r * k: offset // 32 + r * k + len(row)] = row


def _scales_column_major(data_buf, scale_buf, offset, codes, scales):
    c = np.asarray(codes, np.uint8).reshape(-1)
    data_buf[offset: offset + c.size] = c
    s = np.asarray(scales, np.uint8).T.reshape(-1)
    scale_buf[offset // 32: offset // 32 + s.size] = s


@pytest.mark.parametrize("mutant", [_scale_base_at_offset, _scale_stride_k, _scales_column_major])
def test_planted_mistakes_in_the_python_oracle_are_caught(mutant, monkeypatch):
    monkeypatch.setattr(G, "store_mxfp8", mutant)
    with pytest.raises((AssertionError, ValueError)):
        check_fixture(lambda *a: G.run_workload(*a))
