"""Golden reshard semantics in Python + numpy (TEST INFRASTRUCTURE).

Only tests, smoke() and the bench's CPU-baseline leg may use this module; it shares no code
with the CUDA path.

What the reshard computes has a plain definition, given by the debugging transport in the
NeMo-RL design doc "NCCL Reshard Refit (Experimental)", section "xferdtensor Transports":
broadcast the full tensor to the destination ranks, which then drop what they do not own.
This module writes that definition out:

1. every source rank's shard box follows from the DTensor description (global shape, device
   mesh, Shard/Replicate placements; "Execution Flow: Setup Time", and the news article on the
   Reshard collective, section "Recasting refit as a DTensor-to-DTensor transfer");
2. the full tensor is materialised from the source shards, checking that replicas agree and
   that the sources cover every element;
3. every destination rank keeps the slice its own box names, optionally quantized to MXFP8
   ("Enabling It": the generation ranks quantize each received BF16 shard).

Readings of points the pages leave open (each also listed in the design notes):
- uneven split: torch.chunk's rule, chunk c = ceil(L / n), rank i holds
  [min(i c, L), min((i + 1) c, L)); trailing ranks may be empty;
- several mesh dims sharding one tensor dim: mesh dim 0 splits first, each later mesh dim
  chunks the interval left by the earlier ones (DTensor's order);
- ranks are numbered row-major over mesh coordinates;
- among replicated sources, the lowest rank supplies a region (the result does not depend on
  the choice, since replicas must agree).

Parity: pinned by the 8x8 worked example (golden fixture), brute force over small meshes with
element-id payloads, torch.chunk as the library definition of the split, the byte invariants
and the A->B->A round trip; the MXFP8 placement (``store_mxfp8``) by a hand-derived fixture of
where every code and scale byte lands, and against the C oracle (tests).
"""
from __future__ import annotations

import itertools
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import mxfp8 as _mx

NP_DTYPES = {"u8": np.uint8, "bf16": np.uint16, "f16": np.uint16, "f32": np.uint32,
             "i32": np.int32, "i64": np.int64}
ESIZE = {"u8": 1, "bf16": 2, "f16": 2, "f32": 4, "i32": 4, "i64": 8}


def chunk_bounds(length: int, n: int, i: int) -> Tuple[int, int]:
    """[lo, hi) of chunk i when ``length`` is split n ways by torch.chunk's rule."""
    c = -(-length // n) if length > 0 else 0
    return min(i * c, length), min((i + 1) * c, length)


def parse_placement(p: str):
    return ("R",) if p == "R" else ("S", int(p[1:]))


def mesh_coords(mesh: Sequence[int]) -> List[Tuple[int, ...]]:
    """Mesh coordinates in row-major rank order."""
    return list(itertools.product(*[range(int(n)) for n in mesh]))


def shard_box(global_shape: Sequence[int], mesh: Sequence[int], placements: Sequence[str],
              coord: Sequence[int]) -> List[Tuple[int, int]]:
    """Per tensor dim [lo, hi) owned by the rank at ``coord``.

    Mesh dims are applied in order; a Shard(d) on mesh dim k chunks the interval that the
    earlier mesh dims left for tensor dim d into mesh[k] pieces and keeps piece coord[k].
    """
    box = [(0, int(n)) for n in global_shape]
    for k, p in enumerate(placements):
        pl = parse_placement(p)
        if pl[0] == "R":
            continue
        d = pl[1]
        lo, hi = box[d]
        a, b = chunk_bounds(hi - lo, int(mesh[k]), int(coord[k]))
        box[d] = (lo + a, lo + b)
    return box


def box_shape(box) -> Tuple[int, ...]:
    return tuple(hi - lo for lo, hi in box)


def box_numel(box) -> int:
    return int(np.prod(box_shape(box))) if len(box) else 1


def local_array(buf_u8: np.ndarray, dtype: str, offset: int, strides, shape) -> np.ndarray:
    """The local shard as a numpy view into a byte buffer (element offset and strides)."""
    es = ESIZE[dtype]
    typed = buf_u8.view(NP_DTYPES[dtype]) if buf_u8.size else np.zeros(0, NP_DTYPES[dtype])
    if int(np.prod(shape)) == 0:
        return np.zeros(shape, NP_DTYPES[dtype])
    if strides is None:
        strides = [int(np.prod(shape[i + 1:])) for i in range(len(shape))]
    return np.lib.stride_tricks.as_strided(typed[offset:], shape=shape,
                                           strides=[s * es for s in strides], writeable=True)


# ---------------------------------------------------------------------------------------
# golden: materialise the full tensor, then slice every destination
# ---------------------------------------------------------------------------------------

class OracleError(Exception):
    pass


def materialise(desc, src_bufs: Sequence[np.ndarray]) -> np.ndarray:
    """The full global tensor, assembled from every source rank's shard.

    Raises OracleError when two replicas disagree or an element has no source.
    """
    full = np.zeros(tuple(desc.global_shape), NP_DTYPES[desc.dtype])
    have = np.zeros(tuple(desc.global_shape), bool)
    for r, coord in enumerate(mesh_coords(desc.src_mesh)):
        box = shard_box(desc.global_shape, desc.src_mesh, desc.src_placements, coord)
        v = desc.src_views[r]
        loc = local_array(src_bufs[r], desc.dtype, v.offset, v.strides, box_shape(box))
        sl = tuple(slice(lo, hi) for lo, hi in box)
        seen = have[sl]
        if seen.any() and not np.array_equal(full[sl][seen], loc[seen]):
            raise OracleError(f"{desc.name}: source replicas disagree (rank {r})")
        full[sl] = loc
        have[sl] = True
    if not have.all():
        raise OracleError(f"{desc.name}: sources leave {int((~have).sum())} elements uncovered")
    return full


def golden_reshard(desc, src_bufs: Sequence[np.ndarray], dst_bufs: Sequence[np.ndarray],
                   quant: str = "none", scale_bufs: Optional[Sequence[np.ndarray]] = None) -> None:
    """Write every destination rank's shard (in place into its byte buffer)."""
    full = materialise(desc, src_bufs)
    for r, coord in enumerate(mesh_coords(desc.dst_mesh)):
        box = shard_box(desc.global_shape, desc.dst_mesh, desc.dst_placements, coord)
        shp = box_shape(box)
        v = desc.dst_views[r]
        part = full[tuple(slice(lo, hi) for lo, hi in box)]
        if box_numel(box) == 0:
            continue
        if quant == "none":
            local_array(dst_bufs[r], desc.dtype, v.offset, v.strides, shp)[...] = part
            continue
        if desc.dtype != "bf16" or shp[-1] % 32 or v.strides is not None or v.offset % 32:
            raise OracleError(f"{desc.name}: mxfp8 needs bf16, dense views and K % 32 == 0")
        rows = part.reshape(-1, shp[-1])
        codes, scales = _mx.quantize_rows([[int(b) for b in row] for row in rows])
        store_mxfp8(dst_bufs[r], scale_bufs[r], v.offset, codes, scales)


def store_mxfp8(data_buf: np.ndarray, scale_buf: np.ndarray, offset: int, codes, scales) -> None:
    """Place one quantized shard: its E4M3 codes (one byte per element, row-major rows of the
    local shard) from byte ``offset`` of the data buffer, and its E8M0 scales (one byte per
    32-element block, row-major [..., K_local / 32]) from byte ``offset // 32`` of the scale
    buffer. The layout is the plainest reading of "quantize each received shard" ("Enabling
    It") under the OCP MX v1.0 block rule; ``offset`` is a multiple of 32."""
    c = np.asarray(codes, np.uint8).reshape(-1)
    s = np.asarray(scales, np.uint8).reshape(-1)
    data_buf[offset: offset + c.size] = c
    scale_buf[offset // 32: offset // 32 + s.size] = s


def run_workload(wl, src_slab: np.ndarray, src_off, dst_slab: np.ndarray, dst_off,
                 scale_slab: Optional[np.ndarray] = None, scale_off=None) -> None:
    """Golden reshard of every tensor of a synthetic workload, in place on host slabs."""
    for t in wl.tensors:
        es = ESIZE[t.dtype]
        sb = [src_slab[src_off[v.buffer]: src_off[v.buffer] + wl.src_buffer_numel[v.buffer] * es]
              for v in t.src_views]
        if wl.quant == "mxfp8":
            db = [dst_slab[dst_off[v.buffer]: dst_off[v.buffer] + wl.dst_buffer_numel[v.buffer]]
                  for v in t.dst_views]
            cb = [scale_slab[scale_off[v.buffer]: scale_off[v.buffer] + wl.dst_buffer_numel[v.buffer] // 32]
                  for v in t.dst_views]
        else:
            db = [dst_slab[dst_off[v.buffer]: dst_off[v.buffer] + wl.dst_buffer_numel[v.buffer] * es]
                  for v in t.dst_views]
            cb = None
        golden_reshard(t, sb, db, wl.quant, cb)


# ---------------------------------------------------------------------------------------
# brute-force region enumeration and the one-element mapping
# ---------------------------------------------------------------------------------------

def holders(desc, gidx: Sequence[int]) -> List[int]:
    """Every source rank whose box contains global index ``gidx``."""
    out = []
    for r, coord in enumerate(mesh_coords(desc.src_mesh)):
        box = shard_box(desc.global_shape, desc.src_mesh, desc.src_placements, coord)
        if all(lo <= i < hi for i, (lo, hi) in zip(gidx, box)):
            out.append(r)
    return out


def source_regions(desc) -> List[Tuple[Tuple[int, ...], int, Tuple[Tuple[int, int], ...]]]:
    """Brute force: per destination replica group and supplying source, the region it gets.

    Every destination element is assigned the lowest-rank source holding it; the elements a
    (destination group, source) pair exchanges must form one box, which is returned in global
    coordinates. Result: sorted list of (destination ranks of the group, source rank, box).
    For tiny tensors only (pure-Python loops over every element).
    """
    groups: Dict[Tuple[Tuple[int, int], ...], List[int]] = {}
    for r, coord in enumerate(mesh_coords(desc.dst_mesh)):
        box = tuple(shard_box(desc.global_shape, desc.dst_mesh, desc.dst_placements, coord))
        groups.setdefault(box, []).append(r)
    out = []
    for box, members in groups.items():
        per_src: Dict[int, List[Tuple[int, ...]]] = {}
        for gidx in itertools.product(*[range(lo, hi) for lo, hi in box]):
            hs = holders(desc, gidx)
            if not hs:
                raise OracleError("element without a source")
            per_src.setdefault(hs[0], []).append(gidx)
        for s, elems in per_src.items():
            arr = np.array(elems)
            lo = arr.min(axis=0)
            hi = arr.max(axis=0) + 1
            if int(np.prod(hi - lo)) != len(elems):
                raise OracleError("a (destination, source) exchange is not one box")
            out.append((tuple(members), s, tuple((int(a), int(b)) for a, b in zip(lo, hi))))
    return sorted(out)


def dst_element_source(desc, dst_rank: int, local_idx: Sequence[int]) -> Tuple[int, Tuple[int, ...]]:
    """Which source rank and local index hold destination ``dst_rank``'s element ``local_idx``.

    The lowest-rank holder is returned. Used one element at a time for sampled parity.
    """
    dcoord = mesh_coords(desc.dst_mesh)[dst_rank]
    dbox = shard_box(desc.global_shape, desc.dst_mesh, desc.dst_placements, dcoord)
    gidx = tuple(lo + i for (lo, _), i in zip(dbox, local_idx))
    hs = holders(desc, gidx)
    if not hs:
        raise OracleError("element without a source")
    s = hs[0]
    sbox = shard_box(desc.global_shape, desc.src_mesh, desc.src_placements, mesh_coords(desc.src_mesh)[s])
    return s, tuple(g - lo for g, (lo, _) in zip(gidx, sbox))


def element_offset(view, shape: Sequence[int], idx: Sequence[int]) -> int:
    """Element offset inside the buffer of local index ``idx`` under a view."""
    if view.strides is None:
        strides = [int(np.prod(shape[i + 1:])) for i in range(len(shape))]
    else:
        strides = view.strides
    return view.offset + sum(i * s for i, s in zip(idx, strides))


# ---------------------------------------------------------------------------------------
# byte accounting (closed forms on the boxes)
# ---------------------------------------------------------------------------------------

def byte_accounting(desc) -> Dict[str, int]:
    """Bytes the method moves for one tensor, from the boxes alone.

    - written: every destination shard, replicas included ("each generation rank receives
      exactly the bytes of its own shard", design doc introduction);
    - read: each element once per distinct destination box (replica group): "moves each
      destination region once" ("xferdtensor Transports");
    - gather_bcast: the two-stage all-gather + broadcast payload, about twice the tensor
      (news article, "Why refit is challenging in RL post-training").
    """
    es = ESIZE[desc.dtype]
    written = 0
    boxes = set()
    for coord in mesh_coords(desc.dst_mesh):
        box = tuple(shard_box(desc.global_shape, desc.dst_mesh, desc.dst_placements, coord))
        written += box_numel(box) * es
        if box_numel(box):
            boxes.add(box)   # a replica group is a set of ranks sharing one non-empty box
    read = sum(box_numel(b) * es for b in boxes)
    total = int(np.prod(desc.global_shape)) * es
    return {"bytes_written": written, "bytes_read": read, "gather_bcast_bytes": 2 * total,
            "dst_groups": len(boxes)}
