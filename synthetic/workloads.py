"""Synthetic reshard workloads: problem descriptions plus seeded value generators.

A workload is a list of weight tensors, each described the way a DTensor is (global shape,
dtype, device mesh, Shard/Replicate placements) once for the training (source) side and once
for the generation (destination) side, plus how every rank's local shard sits inside a
caller-owned buffer (a "view": buffer index, element offset, optional element strides).

Everything the reshard method computes (shard boxes, intersections, source choice, copies,
quantization) lives elsewhere. The one piece of layout arithmetic used here is the source
layout itself, and it is produced with ``torch.chunk``, which is PyTorch's own definition of a
DTensor ``Shard`` placement, the way a training framework lays its weights out. Local shard
shapes for buffer sizing are taken the same way, on the ``meta`` device.

Workload recipes follow the weight shapes named in "Accelerating RL Weight Refit with the
Reshard Collective" (the 8x8 example) and the NeMo-RL design doc "NCCL Reshard Refit"
(dense FFN projections, grouped MoE experts, fused gate_up on the training side).
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

# name -> (torch dtype, element size in bytes)
DTYPES = {
    "u8": (torch.uint8, 1),
    "bf16": (torch.bfloat16, 2),
    "f16": (torch.float16, 2),
    "f32": (torch.float32, 4),
    "i32": (torch.int32, 4),
    "i64": (torch.int64, 8),
}


@dataclass
class View:
    """Where one rank's local shard lives: buffer index, element offset, element strides.

    ``strides=None`` means dense row-major strides of the local shard shape.
    """
    buffer: int
    offset: int = 0
    strides: Optional[Tuple[int, ...]] = None


@dataclass
class TensorDesc:
    name: str
    global_shape: Tuple[int, ...]
    dtype: str
    src_mesh: Tuple[int, ...]
    src_placements: Tuple[str, ...]   # one per mesh dim: "R" or "S<d>"
    dst_mesh: Tuple[int, ...]
    dst_placements: Tuple[str, ...]
    src_views: List[View]             # one per source rank, row-major over mesh coordinates
    dst_views: List[View]
    seed: int = 0
    std: float = 1.0

    @property
    def n_src(self) -> int:
        return int(np.prod(self.src_mesh))

    @property
    def n_dst(self) -> int:
        return int(np.prod(self.dst_mesh))


@dataclass
class Workload:
    name: str
    tensors: List[TensorDesc]
    quant: str = "none"              # "none" | "mxfp8"
    values: str = "randn"            # "randn" | "iota" | "bytes"
    src_buffer_numel: List[int] = field(default_factory=list)
    src_buffer_dtype: List[str] = field(default_factory=list)
    dst_buffer_numel: List[int] = field(default_factory=list)
    dst_buffer_dtype: List[str] = field(default_factory=list)
    block: Optional[Tuple[int, int]] = None  # blockwise FP8: tensors = weights, then their scales

    def src_bytes(self) -> int:
        return sum(n * DTYPES[d][1] for n, d in zip(self.src_buffer_numel, self.src_buffer_dtype) if n)

    def dst_bytes(self) -> int:
        """Bytes of every destination buffer (data, plus scales under mxfp8)."""
        if self.quant == "mxfp8":
            return sum(n + n // 32 for n in self.dst_buffer_numel)
        return sum(n * DTYPES[d][1] for n, d in zip(self.dst_buffer_numel, self.dst_buffer_dtype) if n)


# ----------------------------------------------------------------------------------------
# local shapes through torch.chunk (PyTorch's definition of a DTensor Shard placement)
# ----------------------------------------------------------------------------------------

def mesh_coords(mesh: Sequence[int]):
    return list(itertools.product(*[range(int(n)) for n in mesh]))


def _chunk_local(t: torch.Tensor, mesh, placements, coord) -> torch.Tensor:
    for k, pl in enumerate(placements):
        if pl == "R":
            continue
        d = int(pl[1:])
        if t.shape[d] == 0:
            t = t.narrow(d, 0, 0)
            continue
        parts = torch.chunk(t, int(mesh[k]), dim=d)
        t = parts[coord[k]] if coord[k] < len(parts) else t.narrow(d, t.shape[d], 0)
    return t


def local_shape(global_shape, mesh, placements, coord) -> Tuple[int, ...]:
    meta = torch.empty(tuple(global_shape), device="meta")
    return tuple(_chunk_local(meta, mesh, placements, coord).shape)


def _need(shape, view: View) -> int:
    n = int(np.prod(shape)) if len(shape) else 1
    if n == 0:
        return view.offset
    if view.strides is None:
        return view.offset + n
    return view.offset + sum((s - 1) * st for s, st in zip(shape, view.strides)) + 1


def _size_buffers(wl: Workload, n_src_buf: int, n_dst_buf: int) -> Workload:
    wl.src_buffer_numel = [0] * n_src_buf
    wl.src_buffer_dtype = [""] * n_src_buf
    wl.dst_buffer_numel = [0] * n_dst_buf
    wl.dst_buffer_dtype = [""] * n_dst_buf
    for t in wl.tensors:
        for side, mesh, pls, views, numel, dts in (
                ("src", t.src_mesh, t.src_placements, t.src_views, wl.src_buffer_numel, wl.src_buffer_dtype),
                ("dst", t.dst_mesh, t.dst_placements, t.dst_views, wl.dst_buffer_numel, wl.dst_buffer_dtype)):
            assert len(views) == int(np.prod(mesh)), (t.name, side)
            for coord, v in zip(mesh_coords(mesh), views):
                shp = local_shape(t.global_shape, mesh, pls, coord)
                numel[v.buffer] = max(numel[v.buffer], _need(shp, v))
                dt = "u8" if (side == "dst" and wl.quant == "mxfp8") else t.dtype
                assert dts[v.buffer] in ("", dt), "one dtype per buffer"
                dts[v.buffer] = dt
    return wl


# ----------------------------------------------------------------------------------------
# workload recipes
# ----------------------------------------------------------------------------------------

def _dense_views(n: int, start: int) -> List[View]:
    return [View(start + i) for i in range(n)]


def example_8x8(seed: int = 1) -> Workload:
    """The 8x8 example: two 4x8 row shards into four 8x2 column shards."""
    t = TensorDesc("w", (8, 8), "bf16", (2,), ("S0",), (4,), ("S1",),
                   _dense_views(2, 0), _dense_views(4, 0), seed=seed, std=1.0)
    return _size_buffers(Workload("example_8x8", [t]), 2, 4)


def dense_ffn(layers: int = 32, hidden: int = 4096, ffn: int = 14336, tp_src: int = 8,
              dp_dst: int = 2, tp_dst: int = 2, seed: int = 2, std: float = 0.02,
              fused: str = "block", dtype: str = "bf16") -> Workload:
    """Dense FFN projections. Training side: Megatron TP with gate/up fused per rank.

    ``fused="block"``: per rank one buffer holding [gate_r; up_r] (rows of gate then rows of up).
    ``fused="interleave"``: per rank one buffer whose rows alternate gate row, up row.
    ``fused="none"``: separate gate and up buffers.
    Generation side: (DP, TP) mesh with [Replicate, Shard], separate gate/up/down buffers.
    """
    tensors: List[TensorDesc] = []
    nsb = 0
    ndb = 0
    n_dst = dp_dst * tp_dst
    for layer in range(layers):
        s = seed * 1_000_003 + layer * 3
        gate_rows = [local_shape((ffn, hidden), (tp_src,), ("S0",), (r,))[0] for r in range(tp_src)]
        if fused == "none":
            gate_v = _dense_views(tp_src, nsb); nsb += tp_src
            up_v = _dense_views(tp_src, nsb); nsb += tp_src
        else:
            fb = list(range(nsb, nsb + tp_src)); nsb += tp_src
            if fused == "block":
                gate_v = [View(fb[r], 0) for r in range(tp_src)]
                up_v = [View(fb[r], gate_rows[r] * hidden) for r in range(tp_src)]
            elif fused == "interleave":
                gate_v = [View(fb[r], 0, (2 * hidden, 1)) for r in range(tp_src)]
                up_v = [View(fb[r], hidden, (2 * hidden, 1)) for r in range(tp_src)]
            else:
                raise ValueError(fused)
        down_v = _dense_views(tp_src, nsb); nsb += tp_src
        dmesh = (dp_dst, tp_dst)
        g_d = _dense_views(n_dst, ndb); ndb += n_dst
        u_d = _dense_views(n_dst, ndb); ndb += n_dst
        d_d = _dense_views(n_dst, ndb); ndb += n_dst
        tensors.append(TensorDesc(f"layers.{layer}.mlp.gate_proj.weight", (ffn, hidden), dtype,
                                  (tp_src,), ("S0",), dmesh, ("R", "S0"), gate_v, g_d, s, std))
        tensors.append(TensorDesc(f"layers.{layer}.mlp.up_proj.weight", (ffn, hidden), dtype,
                                  (tp_src,), ("S0",), dmesh, ("R", "S0"), up_v, u_d, s + 1, std))
        tensors.append(TensorDesc(f"layers.{layer}.mlp.down_proj.weight", (hidden, ffn), dtype,
                                  (tp_src,), ("S1",), dmesh, ("R", "S1"), down_v, d_d, s + 2, std))
    name = f"dense_ffn_{layers}x{ffn}x{hidden}_tp{tp_src}_to_dp{dp_dst}tp{tp_dst}"
    return _size_buffers(Workload(name, tensors), nsb, ndb)


def moe_experts(layers: int = 8, experts: int = 128, hidden: int = 4096, ffn: int = 1536,
                ep_src: int = 16, dst: str = "ep8", seed: int = 3, std: float = 0.02) -> Workload:
    """Grouped MoE expert weights [E, ffn, hidden] (gate, up) and [E, hidden, ffn] (down).

    Training side: EP over the expert dim (ETP=1, each rank holds whole experts).
    ``dst="ep<N>"``: generation EP=N over the expert dim, BF16.
    ``dst="tp<N>"``: generation TP=N (gate/up split on ffn rows, down on the ffn input dim),
    received as MXFP8 (E4M3 data + E8M0 scale per 32 elements along the last dim).
    """
    tensors: List[TensorDesc] = []
    nsb = ndb = 0
    kind, n = dst[:2], int(dst[2:])
    quant = "mxfp8" if kind == "tp" else "none"
    for layer in range(layers):
        s = seed * 1_000_003 + layer * 3
        for j, (proj, shape) in enumerate((("gate_proj", (experts, ffn, hidden)),
                                           ("up_proj", (experts, ffn, hidden)),
                                           ("down_proj", (experts, hidden, ffn)))):
            sv = _dense_views(ep_src, nsb); nsb += ep_src
            dv = _dense_views(n, ndb); ndb += n
            if kind == "ep":
                dpl = ("S0",)
            else:
                dpl = ("S1",) if proj != "down_proj" else ("S2",)
            tensors.append(TensorDesc(f"layers.{layer}.mlp.experts.{proj}.weight", shape, "bf16",
                                      (ep_src,), ("S0",), (n,), dpl, sv, dv, s + j, std))
    name = f"moe_{layers}x{experts}x{ffn}x{hidden}_ep{ep_src}_to_{dst}" + ("_mxfp8" if quant == "mxfp8" else "")
    return _size_buffers(Workload(name, tensors, quant=quant), nsb, ndb)


def uneven_tp(rows: int = 14336, cols: int = 4096, src: int = 6, dst: int = 5, seed: int = 5,
              dtype: str = "bf16") -> Workload:
    """One tensor with uneven torch.chunk splits: TP=src rows into TP=dst rows."""
    t = TensorDesc("w", (rows, cols), dtype, (src,), ("S0",), (dst,), ("S0",),
                   _dense_views(src, 0), _dense_views(dst, 0), seed=seed, std=1.0)
    return _size_buffers(Workload(f"uneven_{rows}x{cols}_tp{src}_to_tp{dst}", [t]), src, dst)


def mesh2d_to_1d(rows: int = 14336, cols: int = 4096, variant: str = "1d", seed: int = 5,
                 dtype: str = "bf16", src_cols: int = 4) -> Workload:
    """A (2, src_cols) [Shard(0), Shard(1)] source into a 3-way column split.

    ``variant="1d"``: destination mesh (3,) [Shard(1)]; ``"2d"``: (3,2) [Shard(1), Replicate].
    """
    if variant == "1d":
        dmesh, dpl = (3,), ("S1",)
    else:
        dmesh, dpl = (3, 2), ("S1", "R")
    nd = int(np.prod(dmesh))
    ns = 2 * src_cols
    t = TensorDesc("w", (rows, cols), dtype, (2, src_cols), ("S0", "S1"), dmesh, dpl,
                   _dense_views(ns, 0), _dense_views(nd, 0), seed=seed, std=1.0)
    return _size_buffers(Workload(f"mesh2x{src_cols}_to_{'x'.join(map(str, dmesh))}_{rows}x{cols}", [t]), ns, nd)


def many_small(n: int = 10000, size_seed: int = 55, value_seed: int = 56, rows=(64, 512),
               cols=(64, 4096), tp_src: int = 4, dp_dst: int = 2, tp_dst: int = 2) -> Workload:
    """Many small BF16 tensors with seeded shapes, TP row split into (DP, TP) [Replicate, Shard(0)]."""
    rng = np.random.Generator(np.random.PCG64(size_seed))
    r = rng.integers(rows[0], rows[1] + 1, size=n)
    c = rng.integers(cols[0], cols[1] + 1, size=n)
    tensors = []
    nsb = ndb = 0
    nd = dp_dst * tp_dst
    for i in range(n):
        sv = _dense_views(tp_src, nsb); nsb += tp_src
        dv = _dense_views(nd, ndb); ndb += nd
        tensors.append(TensorDesc(f"t{i}", (int(r[i]), int(c[i])), "bf16", (tp_src,), ("S0",),
                                  (dp_dst, tp_dst), ("R", "S0"), sv, dv,
                                  seed=value_seed * 1_000_003 + i, std=1.0))
    return _size_buffers(Workload(f"many_small_{n}_tp{tp_src}_to_dp{dp_dst}tp{tp_dst}", tensors), nsb, ndb)


def _colmajor_views(global_shape, mesh, placements, start: int) -> List[View]:
    """Views that store each local shard with its last two dims transposed (dim -2 contiguous)."""
    out = []
    for i, coord in enumerate(mesh_coords(mesh)):
        shp = local_shape(global_shape, mesh, placements, coord)
        nd = len(shp)
        st = [0] * nd
        st[-2] = 1
        st[-1] = max(1, shp[-2])
        acc = max(1, shp[-2]) * max(1, shp[-1])
        for d in range(nd - 3, -1, -1):
            st[d] = acc
            acc *= max(1, shp[d])
        out.append(View(start + i, 0, tuple(st)))
    return out


def transposed(shape=(14336, 4096), src_mesh=(8,), src_pl=("S0",), dst_mesh=(2, 2), dst_pl=("R", "S0"),
               side: str = "dst", dtype: str = "bf16", seed: int = 6, std: float = 0.02, tensors: int = 1) -> Workload:
    """Tensors whose local shards are stored with the last two dims transposed on one side
    (``side="dst"``: the generation side keeps W^T; ``"src"``: the training side does; ``"both"``)."""
    ts = []
    nsb = ndb = 0
    ns, nd = int(np.prod(src_mesh)), int(np.prod(dst_mesh))
    for k in range(tensors):
        sv = _colmajor_views(shape, src_mesh, src_pl, nsb) if side in ("src", "both") else _dense_views(ns, nsb)
        dv = _colmajor_views(shape, dst_mesh, dst_pl, ndb) if side in ("dst", "both") else _dense_views(nd, ndb)
        nsb += ns
        ndb += nd
        ts.append(TensorDesc(f"w{k}", tuple(shape), dtype, tuple(src_mesh), tuple(src_pl), tuple(dst_mesh),
                             tuple(dst_pl), sv, dv, seed=seed * 1_000_003 + k, std=std))
    name = (f"transpose_{tensors}x{'x'.join(map(str, shape))}_{'x'.join(map(str, src_mesh))}{''.join(src_pl)}_to_"
            f"{'x'.join(map(str, dst_mesh))}{''.join(dst_pl)}_{side}_colmajor")
    return _size_buffers(Workload(name, ts), nsb, ndb)


def large_offsets(rows: int = 65536, cols: int = 49152, seed: int = 9, transposing: bool = True) -> Workload:
    """Buffers of more than 2^31 elements on both sides, so that element offsets need 64 bits:
    one replica into a 2-way column split, a 2-way column split back into one replica, and
    (``transposing``) a 2-way row split into one column-major replica."""
    ts = [
        TensorDesc("rep_to_tp2", (rows, cols), "bf16", (1,), ("R",), (2,), ("S1",),
                   _dense_views(1, 0), _dense_views(2, 0), seed=seed, std=1.0),
        TensorDesc("tp2_to_rep", (rows, cols), "bf16", (2,), ("S1",), (1,), ("R",),
                   _dense_views(2, 1), _dense_views(1, 2), seed=seed + 1, std=1.0),
    ]
    nsb, ndb = 3, 3
    if transposing:
        ts.append(TensorDesc("tp2_to_rep_colmajor", (rows, cols), "bf16", (2,), ("S0",), (1,), ("R",),
                             _dense_views(2, 3), _colmajor_views((rows, cols), (1,), ("R",), 3),
                             seed=seed + 2, std=1.0))
        nsb, ndb = 5, 4
    return _size_buffers(Workload(f"large_offsets_{rows}x{cols}", ts), nsb, ndb)


def qkv_kv_below_tp(layers: int = 4, q_heads: int = 64, kv_heads: int = 2, head_dim: int = 128,
                    hidden: int = 8192, tp_src: int = 8, tp_dst: int = 8, seed: int = 8, std: float = 0.02) -> Workload:
    """Fused QKV projections with fewer KV heads than TP ranks, on both sides.

    Each rank's fused buffer holds [q rows; k rows; v rows] of its heads. Q rows are Shard(0)
    over TP. With KV heads below TP, K and V are split over KV groups of TP ranks and replicated
    inside a group, i.e. a (kv, tp / kv) mesh with [Shard(0), Replicate] in the same rank order
    (the ModelExpress reshard PR: "Nemotron-style layers can have fewer KV heads than TP ranks").
    """
    tensors: List[TensorDesc] = []
    nsb = ndb = 0

    def side(tp):
        if kv_heads >= tp:
            return (tp,), ("S0",)
        return (kv_heads, tp // kv_heads), ("S0", "R")

    for layer in range(layers):
        s = seed * 1_000_003 + layer * 3
        ql_src, ql_dst = q_heads // tp_src * head_dim, q_heads // tp_dst * head_dim
        kvl_src = max(1, kv_heads // tp_src) * head_dim
        kvl_dst = max(1, kv_heads // tp_dst) * head_dim
        fs = list(range(nsb, nsb + tp_src)); nsb += tp_src
        fd = list(range(ndb, ndb + tp_dst)); ndb += tp_dst
        kvm_s, kvp_s = side(tp_src)
        kvm_d, kvp_d = side(tp_dst)
        for j, (nm, rows, off_s, off_d, ms, ps, md, pd) in enumerate((
                ("q_proj", q_heads * head_dim, 0, 0, (tp_src,), ("S0",), (tp_dst,), ("S0",)),
                ("k_proj", kv_heads * head_dim, ql_src, ql_dst, kvm_s, kvp_s, kvm_d, kvp_d),
                ("v_proj", kv_heads * head_dim, ql_src + kvl_src, ql_dst + kvl_dst, kvm_s, kvp_s, kvm_d, kvp_d))):
            sv = [View(fs[r], off_s * hidden) for r in range(tp_src)]
            dv = [View(fd[r], off_d * hidden) for r in range(tp_dst)]
            tensors.append(TensorDesc(f"layers.{layer}.self_attn.{nm}.weight", (rows, hidden), "bf16",
                                      ms, ps, md, pd, sv, dv, s + j, std))
    name = f"qkv_{layers}x{q_heads}q{kv_heads}kv{head_dim}x{hidden}_tp{tp_src}_to_tp{tp_dst}"
    return _size_buffers(Workload(name, tensors), nsb, ndb)


def moe_w13(layers: int = 2, experts: int = 64, hidden: int = 2048, ffn: int = 768, ep_src: int = 8,
            tp_dst: int = 4, per_expert_src: bool = True, seed: int = 9, std: float = 0.02) -> Workload:
    """MoE experts into vLLM's fused layout: per rank w13 [E, 2 I_local, H] (gate rows then up
    rows of each expert) and w2 [E, H, I_local], TP over the expert FFN dim.

    ``per_expert_src``: the training side keeps every expert's gate/up/down in its own
    allocation (no stacking copy): each expert is its own tensor [1, ...] whose source mesh is
    the single rank that owns it, and whose destination views point into the fused buffers.
    Otherwise the source is the grouped [E, ...] tensor over EP (stacked).
    """
    tensors: List[TensorDesc] = []
    nsb = ndb = 0
    il = ffn // tp_dst
    for layer in range(layers):
        s = seed * 1_000_003 + layer * 1000
        w13 = list(range(ndb, ndb + tp_dst)); ndb += tp_dst
        w2 = list(range(ndb, ndb + tp_dst)); ndb += tp_dst
        st13 = (2 * il * hidden, hidden, 1)
        if per_expert_src:
            for e in range(experts):
                for j, (nm, shape) in enumerate((("gate_proj", (1, ffn, hidden)), ("up_proj", (1, ffn, hidden)),
                                                 ("down_proj", (1, hidden, ffn)))):
                    sv = [View(nsb)]; nsb += 1
                    if nm == "down_proj":
                        dv = [View(w2[r], e * hidden * il) for r in range(tp_dst)]
                        dpl = ("S2",)
                    else:
                        base = e * 2 * il * hidden + (il * hidden if nm == "up_proj" else 0)
                        dv = [View(w13[r], base, st13) for r in range(tp_dst)]
                        dpl = ("S1",)
                    tensors.append(TensorDesc(f"layers.{layer}.mlp.experts.{e}.{nm}.weight", shape, "bf16",
                                              (1,), ("R",), (tp_dst,), dpl, sv, dv, s + 3 * e + j, std))
        else:
            for j, (nm, shape) in enumerate((("gate_proj", (experts, ffn, hidden)), ("up_proj", (experts, ffn, hidden)),
                                             ("down_proj", (experts, hidden, ffn)))):
                sv = _dense_views(ep_src, nsb); nsb += ep_src
                if nm == "down_proj":
                    dv = [View(w2[r]) for r in range(tp_dst)]
                    dpl = ("S2",)
                else:
                    dv = [View(w13[r], il * hidden if nm == "up_proj" else 0, st13) for r in range(tp_dst)]
                    dpl = ("S1",)
                tensors.append(TensorDesc(f"layers.{layer}.mlp.experts.{nm}.weight", shape, "bf16",
                                          (ep_src,), ("S0",), (tp_dst,), dpl, sv, dv, s + j, std))
    src = "per_expert" if per_expert_src else f"ep{ep_src}"
    name = f"moe_w13_{layers}x{experts}x{ffn}x{hidden}_{src}_to_tp{tp_dst}"
    return _size_buffers(Workload(name, tensors), nsb, ndb)


def moe_fp8_blockwise(layers: int = 8, experts: int = 128, hidden: int = 2048, ffn: int = 768, ep_src: int = 8,
                      dp_src: int = 2, tp_dst: int = 2, dp_dst: int = 8, block=(128, 128), seed: int = 10) -> Workload:
    """Blockwise-FP8 MoE experts with their fp32 scales (one per block of the last two dims).

    Training side (DP, EP) [Replicate, Shard(0)]; generation side (DP, TP) [Replicate, Shard]
    with gate/up split on the FFN rows and down on the FFN columns, as the design doc's FP8 row
    (EP8 x DP2 -> TP2 x DP8). Weights are random bytes; the scale tensors' shapes are the weight
    shapes ceil-divided by the block.
    """
    data, scales = [], []
    nsb = ndb = 0
    ns, nd = dp_src * ep_src, dp_dst * tp_dst
    for layer in range(layers):
        s = seed * 1_000_003 + layer * 6
        for j, (nm, shape) in enumerate((("gate_proj", (experts, ffn, hidden)), ("up_proj", (experts, ffn, hidden)),
                                         ("down_proj", (experts, hidden, ffn)))):
            dpl = ("R", "S2") if nm == "down_proj" else ("R", "S1")
            sshape = shape[:-2] + tuple(-(-x // b) for x, b in zip(shape[-2:], block))
            for arr, shp, dt, tag in ((data, shape, "u8", "weight"), (scales, sshape, "f32", "weight_scale_inv")):
                sv = _dense_views(ns, nsb); nsb += ns
                dv = _dense_views(nd, ndb); ndb += nd
                arr.append(TensorDesc(f"layers.{layer}.mlp.experts.{nm}.{tag}", shp, dt, (dp_src, ep_src), ("R", "S0"),
                                      (dp_dst, tp_dst), dpl, sv, dv, s + 2 * j + (tag != "weight"), 1.0))
    name = f"moe_fp8_{layers}x{experts}x{ffn}x{hidden}_dp{dp_src}ep{ep_src}_to_dp{dp_dst}tp{tp_dst}_b{block[0]}x{block[1]}"
    wl = Workload(name, data + scales, block=tuple(block))
    return _size_buffers(wl, nsb, ndb)


def fuzz_cases(n_cases: int, seed: int = 13, max_len: int = 300) -> List[Workload]:
    """Random problems with random buffer layouts: per rank a dense, padded-pitch, column-major
    (last two dims swapped) or offset view, over 2-D/3-D tensors, 1-D/2-D meshes and four dtypes.
    Values are seeded random numbers of the dtype."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for k in range(n_cases):
        nd = int(rng.integers(2, 4))
        shape = tuple(int(x) for x in rng.integers(1, max_len + 1, size=nd))
        if nd == 3:
            shape = (int(rng.integers(1, 5)),) + shape[1:]
        dtype = str(rng.choice(["bf16", "f32", "u8", "i64"]))

        def mesh_and_pl():
            md = int(rng.integers(1, 3))
            mesh = tuple(int(x) for x in rng.integers(1, 5, size=md))
            pls = tuple("R" if c == nd else f"S{c}" for c in rng.integers(0, nd + 1, size=md))
            return mesh, pls

        sm, sp = mesh_and_pl()
        dm, dp = mesh_and_pl()
        views = {}
        nbuf = {"src": 0, "dst": 0}
        for side, mesh, pls in (("src", sm, sp), ("dst", dm, dp)):
            vs = []
            for coord in mesh_coords(mesh):
                shp = local_shape(shape, mesh, pls, coord)
                kind = int(rng.integers(0, 4))
                off = int(rng.integers(0, 9)) if rng.random() < 0.3 else 0
                st = None
                if kind == 1:    # padded row pitch
                    pad = int(rng.integers(1, 40))
                    st = [0] * nd
                    st[-1] = 1
                    st[-2] = max(1, shp[-1]) + pad
                    if nd == 3:
                        st[0] = st[-2] * max(1, shp[-2])
                    st = tuple(st)
                elif kind == 2:  # column-major in the last two dims
                    st = [0] * nd
                    st[-2] = 1
                    st[-1] = max(1, shp[-2])
                    if nd == 3:
                        st[0] = max(1, shp[-2]) * max(1, shp[-1])
                    st = tuple(st)
                vs.append(View(nbuf[side], off, st))
                nbuf[side] += 1
            views[side] = vs
        t = TensorDesc(f"fz{k}", shape, dtype, sm, sp, dm, dp, views["src"], views["dst"], seed=seed * 7919 + k)
        out.append(_size_buffers(Workload(f"fuzz_{k}", [t]), nbuf["src"], nbuf["dst"]))
    return out


def brute_force_cases(n_cases: int, seed: int = 7, max_mesh_dims: int = 3, max_mesh: int = 4,
                      max_tensor_dims: int = 3, max_len: int = 9, dtype: str = "i32") -> List[Workload]:
    """Random small problems: every placement kind, nested mesh dims, uneven and empty chunks.

    Values are element ids ("iota"), so every destination element names its global index.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for k in range(n_cases):
        nd = int(rng.integers(1, max_tensor_dims + 1))
        shape = tuple(int(x) for x in rng.integers(1, max_len + 1, size=nd))

        def mesh_and_pl():
            md = int(rng.integers(1, max_mesh_dims + 1))
            mesh = tuple(int(x) for x in rng.integers(1, max_mesh + 1, size=md))
            pls = []
            for _ in range(md):
                c = int(rng.integers(0, nd + 1))
                pls.append("R" if c == nd else f"S{c}")
            return mesh, tuple(pls)

        sm, sp = mesh_and_pl()
        dm, dp = mesh_and_pl()
        ns, ndst = int(np.prod(sm)), int(np.prod(dm))
        t = TensorDesc(f"bf{k}", shape, dtype, sm, sp, dm, dp,
                       _dense_views(ns, 0), _dense_views(ndst, 0), seed=seed * 1000 + k)
        wl = Workload(f"brute_{k}", [t], values="iota")
        out.append(_size_buffers(wl, ns, ndst))
    return out


WORKLOAD_NAMES = {
    "example_8x8": lambda: example_8x8(),
    "dense_ffn_32x14336x4096_tp8_to_dp2tp2": lambda: dense_ffn(),
    "moe_8x128x1536x4096_ep16_to_ep8": lambda: moe_experts(dst="ep8"),
    "moe_8x128x1536x4096_ep16_to_tp4_mxfp8": lambda: moe_experts(dst="tp4"),
    "uneven_14336x4096_tp6_to_tp5": lambda: uneven_tp(),
    "mesh2x4_to_3_14336x4096": lambda: mesh2d_to_1d(variant="1d"),
    "mesh2x4_to_3x2_14336x4096": lambda: mesh2d_to_1d(variant="2d"),
    "many_small_10000_tp4_to_dp2tp2": lambda: many_small(),
    # reduced layer counts of the same shapes, for profiler captures (a few GB on the device)
    "dense_ffn_4x14336x4096_tp8_to_dp2tp2": lambda: dense_ffn(layers=4),
    "dense_ffn_2x14336x4096_tp8_to_dp2tp2": lambda: dense_ffn(layers=2),
    "many_small_1000_tp4_to_dp2tp2": lambda: many_small(n=1000),
    # KV heads below TP (Q=64, KV=2, head_dim 128) and vLLM fused expert layouts
    "qkv_4x64q2kv128x8192_tp8_to_tp8": lambda: qkv_kv_below_tp(),
    "qkv_32x64q2kv128x8192_tp8_to_tp4": lambda: qkv_kv_below_tp(layers=32, tp_dst=4),
    "moe_w13_48x128x768x2048_ep8_to_tp4": lambda: moe_w13(layers=48, experts=128, per_expert_src=False),
    "moe_w13_4x128x768x2048_per_expert_to_tp4": lambda: moe_w13(layers=4, experts=128, per_expert_src=True),
    "moe_fp8_8x128x768x2048_dp2ep8_to_dp8tp2_b128x128": lambda: moe_fp8_blockwise(),
    "moe_1x32x1536x4096_ep16_to_tp4_mxfp8": lambda: moe_experts(layers=1, experts=32, dst="tp4"),
    # a generation side that keeps every FFN weight transposed (local shards column-major)
    "transpose_32x14336x4096_tp8_to_dp2tp2_dst_colmajor": lambda: transposed(tensors=32),
    "transpose_2x14336x4096_tp8_to_dp2tp2_dst_colmajor": lambda: transposed(tensors=2),
    # a training side that keeps every weight transposed (source shards column-major)
    "transpose_32x14336x4096_tp8_to_dp2tp2_src_colmajor": lambda: transposed(tensors=32, side="src"),
    "moe_1x128x1536x4096_ep16_to_ep8": lambda: moe_experts(layers=1, dst="ep8"),
    "moe_1x32x1536x4096_ep16_to_ep8": lambda: moe_experts(layers=1, experts=32, dst="ep8"),
    # the (2,4) -> (3,) mesh reshard at 4x the rows (470 MB each way, above the 129 MB L2)
    "mesh2x4_to_3_57344x4096": lambda: mesh2d_to_1d(rows=57344, variant="1d"),
    "mesh2x4_to_3x2_57344x4096": lambda: mesh2d_to_1d(rows=57344, variant="2d"),
    # the same destination split from a (2,1) source: each destination row comes from one region
    "mesh2x1_to_3_14336x4096": lambda: mesh2d_to_1d(variant="1d", src_cols=1),
    "mesh2x1_to_3_57344x4096": lambda: mesh2d_to_1d(rows=57344, variant="1d", src_cols=1),
    "moe_1x128x1536x4096_ep16_to_tp4_mxfp8": lambda: moe_experts(layers=1, dst="tp4"),
    # buffers of more than 2^31 elements (64-bit element offsets)
    "large_offsets_65536x49152": lambda: large_offsets(),
}


def workload_by_name(name: str) -> Workload:
    return WORKLOAD_NAMES[name]()


# ----------------------------------------------------------------------------------------
# buffers: slabs carved into caller-owned buffers, seeded values, canary fill
# ----------------------------------------------------------------------------------------

@dataclass
class Layout:
    """Source / destination / scale slabs (uint8 tensors) and each buffer's byte offset."""
    src_slab: torch.Tensor
    dst_slab: torch.Tensor
    scale_slab: Optional[torch.Tensor]
    src_off: List[int]
    dst_off: List[int]
    scale_off: Optional[List[int]]

    def src_ptrs(self, wl: Workload, t: int) -> List[int]:
        base = self.src_slab.data_ptr()
        return [base + self.src_off[v.buffer] for v in wl.tensors[t].src_views]

    def dst_ptrs(self, wl: Workload, t: int) -> List[int]:
        """Destination pointers of tensor t; under mxfp8 a (data, scales) pair per rank."""
        base = self.dst_slab.data_ptr()
        out = []
        for v in wl.tensors[t].dst_views:
            out.append(base + self.dst_off[v.buffer])
            if self.scale_slab is not None:
                out.append(self.scale_slab.data_ptr() + self.scale_off[v.buffer])
        return out

    def all_src_ptrs(self, wl: Workload) -> List[int]:
        return [p for t in range(len(wl.tensors)) for p in self.src_ptrs(wl, t)]

    def all_dst_ptrs(self, wl: Workload) -> List[int]:
        return [p for t in range(len(wl.tensors)) for p in self.dst_ptrs(wl, t)]


def _carve(sizes: List[int], align: int, misalign: int) -> Tuple[List[int], int]:
    offs, cur = [], 0
    for n in sizes:
        off = ((cur + align - 1) // align) * align + misalign
        offs.append(off)
        cur = off + n
    return offs, ((cur + align - 1) // align) * align + align


def allocate(wl: Workload, device, align: int = 256, misalign: int = 0, pin: bool = False) -> Layout:
    """Carve every buffer out of one slab per side. ``misalign`` shifts each buffer's start
    by that many bytes past an ``align`` boundary (to exercise unaligned pointers)."""
    sb = [n * DTYPES[d][1] if n else 0 for n, d in zip(wl.src_buffer_numel, wl.src_buffer_dtype)]
    if wl.quant == "mxfp8":
        db = list(wl.dst_buffer_numel)
    else:
        db = [n * DTYPES[d][1] if n else 0 for n, d in zip(wl.dst_buffer_numel, wl.dst_buffer_dtype)]
    so, stot = _carve(sb, align, misalign)
    do, dtot = _carve(db, align, misalign)
    kw = dict(dtype=torch.uint8, device=device)
    if pin:
        kw["pin_memory"] = True
    src = torch.empty(stot, **kw)
    dst = torch.empty(dtot, **kw)
    scale = None
    sco = None
    if wl.quant == "mxfp8":
        sco, sctot = _carve([n // 32 for n in wl.dst_buffer_numel], align, 0)
        scale = torch.empty(sctot, **kw)
    return Layout(src, dst, scale, so, do, sco)


def _typed(slab: torch.Tensor, byte_off: int, numel: int, dtype: str) -> torch.Tensor:
    tdt, es = DTYPES[dtype]
    return slab[byte_off: byte_off + numel * es].view(tdt)


def _global_values(t: TensorDesc, values: str, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(t.seed))
    tdt, _ = DTYPES[t.dtype]
    if values == "iota":
        n = int(np.prod(t.global_shape))
        return torch.arange(n, dtype=torch.int64, device=device).reshape(t.global_shape).to(tdt)
    if values == "bytes" or t.dtype == "u8":
        return torch.randint(0, 256, t.global_shape, generator=g, device=device, dtype=torch.int64).to(tdt)
    if t.dtype in ("i32", "i64"):
        return torch.randint(-2**31, 2**31 - 1, t.global_shape, generator=g, device=device,
                             dtype=torch.int64).to(tdt)
    x = torch.randn(t.global_shape, generator=g, device=device, dtype=torch.float32)
    return x.mul_(t.std).to(tdt)


def fill_sources(wl: Workload, lay: Layout) -> None:
    """Write every source rank's shard of every tensor into its buffer view."""
    device = lay.src_slab.device
    for t in wl.tensors:
        glob = _global_values(t, wl.values, device)
        for coord, v in zip(mesh_coords(t.src_mesh), t.src_views):
            part = _chunk_local(glob, t.src_mesh, t.src_placements, coord)
            if part.numel() == 0:
                continue
            buf = _typed(lay.src_slab, lay.src_off[v.buffer], wl.src_buffer_numel[v.buffer], t.dtype)
            strides = v.strides if v.strides is not None else torch.empty(part.shape, device="meta").stride()
            torch.as_strided(buf, part.shape, strides, buf.storage_offset() + v.offset).copy_(part)
        del glob


def fill_canary(lay: Layout, byte: int = 0xA5) -> None:
    """Fill destination (and scale) slabs with a known byte so untouched bytes are checkable."""
    lay.dst_slab.fill_(byte)
    if lay.scale_slab is not None:
        lay.scale_slab.fill_(byte)
