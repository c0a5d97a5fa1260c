"""Planted mistakes in the oracle (on the CPU): each must make one of its pins fail."""
from fractions import Fraction

import pytest

from oracle import golden as G
from oracle import mxfp8 as M

import test_oracle_golden as TG
import test_oracle_mxfp8 as TM


def test_floor_split_is_caught():
    def floor_chunk(length, n, i):
        c = length // n
        return min(i * c, length), min((i + 1) * c, length)
    with pytest.raises(AssertionError):
        TG.check_chunk_rule(floor_chunk)


def test_reversed_mesh_order_is_caught():
    orig = G.shard_box

    def reversed_order(global_shape, mesh, placements, coord):
        return orig(global_shape, tuple(reversed(mesh)), tuple(reversed(placements)), tuple(reversed(coord)))
    with pytest.raises(AssertionError):
        TG.check_nested_boxes(reversed_order)


def test_transposed_shard_dim_is_caught(monkeypatch):
    orig = G.shard_box

    def swapped(global_shape, mesh, placements, coord):
        flip = {"S0": "S1", "S1": "S0"}
        return orig(global_shape, mesh, tuple(flip.get(p, p) for p in placements), coord)
    monkeypatch.setattr(G, "shard_box", swapped)
    with pytest.raises(AssertionError):
        TG.check_example_8x8(G.source_regions, G.golden_reshard)


def test_dropped_replica_check_is_caught(monkeypatch):
    # an oracle that reads source rank 0 for every element gets the 8x8 values wrong
    orig = G.mesh_coords
    monkeypatch.setattr(G, "mesh_coords", lambda mesh: orig(mesh)[:1] * len(orig(mesh)))
    with pytest.raises(Exception):
        TG.check_example_8x8(G.source_regions, G.golden_reshard)


def test_scale_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(M, "E4M3_EMAX", 7)
    with pytest.raises(AssertionError):
        TM.check_block_closed_forms(M.quantize_block)


def test_round_half_up_is_caught():
    def half_up(bits, x):
        v = M.bf16_value(bits) / (Fraction(2) ** x)
        a = abs(v)
        if a == 0:
            return 0x80 if bits >> 15 else 0
        q = M.E4M3_SUB_QUANTUM if a < M.E4M3_MIN_NORMAL else Fraction(2) ** (M.floor_log2(a) - 3)
        k = int(a / q + Fraction(1, 2))
        return M.e4m3_encode(k * q, bool(bits >> 15))
    with pytest.raises(AssertionError):
        TM.check_elements(half_up, stride=29, xs=(0,))
