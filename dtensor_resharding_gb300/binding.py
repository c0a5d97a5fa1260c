"""Thin ctypes binding of libreshard.so: the C-ABI calls under the same names.

Argument marshalling only: every step of the reshard (planning, copies, quantization) runs in
the library. There is no fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Any, Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libreshard.so")

RESHARD_OK = 0
RESHARD_ERR_INVALID_ARG = -1
RESHARD_ERR_UNSUPPORTED = -2
RESHARD_ERR_CUDA = -3
RESHARD_ERR_OOM = -4
RESHARD_ERR_COVERAGE = -5
RESHARD_REPLICATE = 0
RESHARD_SHARD = 1
RESHARD_DIRECT = 0
RESHARD_PACKED = 1
RESHARD_QUANT_NONE = 0
RESHARD_QUANT_MXFP8 = 1
RESHARD_MAX_DIMS = 4
DTYPE_CODES = {"u8": 0, "bf16": 1, "f16": 2, "f32": 3, "i32": 4, "i64": 5}
MODES = {"direct": RESHARD_DIRECT, "packed": RESHARD_PACKED}
QUANTS = {"none": RESHARD_QUANT_NONE, "mxfp8": RESHARD_QUANT_MXFP8}
RESHARD_STRIPED = 1
RESHARD_SEND = 0
RESHARD_RECV = 1
RESHARD_SEND_BUF = 0
RESHARD_RECV_BUF = 1
EXPORTED = ("reshard_plan_create", "reshard_plan_batch", "reshard_plan_blockwise_fp8", "reshard_execute",
            "reshard_execute_pack", "reshard_execute_unpack", "reshard_plan_partition", "reshard_plan_transfers",
            "reshard_execute_static",
            "reshard_plan_stats",
            "reshard_plan_regions", "reshard_plan_group_members", "reshard_plan_items", "reshard_plan_slabs",
            "reshard_plan_status", "reshard_plan_destroy", "reshard_last_error")

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)


class MeshT(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int), ("shape", _i64p), ("ranks", _i32p)]


class PlacementT(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("dim", ctypes.c_int)]


class ViewT(ctypes.Structure):
    _fields_ = [("offset_elems", ctypes.c_int64), ("strides_elems", _i64p), ("capacity_elems", ctypes.c_int64)]


class TensorSpecT(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int), ("global_shape", _i64p), ("dtype", ctypes.c_int),
                ("src_mesh", MeshT), ("src_pl", ctypes.POINTER(PlacementT)), ("src_views", ctypes.POINTER(ViewT)),
                ("dst_mesh", MeshT), ("dst_pl", ctypes.POINTER(PlacementT)), ("dst_views", ctypes.POINTER(ViewT))]


STATS_FIELDS = ("n_tensors", "regions", "items", "dst_groups", "messages", "bytes_read", "bytes_written",
                "wire_bytes", "message_bytes", "gather_bcast_bytes", "global_bytes", "last_launches",
                "last_aligned_items", "last_general_items", "last_rows_kernel", "recv_bytes", "rank", "world",
                "transfers", "sent_bytes", "forwarded_bytes", "local_bytes", "last_staged_items", "gather_items",
                "last_gather_items")


class StatsT(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in STATS_FIELDS]


class TransferT(ctypes.Structure):
    _fields_ = [("peer", ctypes.c_int32), ("dir", ctypes.c_int32), ("buf", ctypes.c_int32), ("phase", ctypes.c_int32),
                ("offset", ctypes.c_int64), ("bytes", ctypes.c_int64)]


class ReshardError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"reshard error {code}: {msg}")
        self.code = code


def _load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libreshard.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.reshard_plan_create.argtypes = [ctypes.POINTER(TensorSpecT), ctypes.POINTER(vp)]
    lib.reshard_plan_batch.argtypes = [ctypes.POINTER(TensorSpecT), ctypes.c_int, ctypes.POINTER(vp)]
    lib.reshard_plan_blockwise_fp8.argtypes = [ctypes.POINTER(TensorSpecT), ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.POINTER(vp)]
    lib.reshard_execute.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int, vp]
    lib.reshard_execute_static.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]
    lib.reshard_execute_pack.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, ctypes.c_int, vp]
    lib.reshard_execute_unpack.argtypes = [vp, vp, ctypes.POINTER(vp), ctypes.c_int, vp]
    lib.reshard_plan_partition.argtypes = [vp, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(vp)]
    lib.reshard_plan_transfers.argtypes = [vp, ctypes.c_int, ctypes.c_int64, ctypes.POINTER(TransferT), _i64p]
    lib.reshard_plan_stats.argtypes = [vp, ctypes.POINTER(StatsT)]
    lib.reshard_plan_regions.argtypes = [vp, ctypes.c_int64, _i32p, _i32p, _i32p, _i64p, _i64p, _i64p]
    lib.reshard_plan_group_members.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, _i32p, _i64p]
    lib.reshard_plan_items.argtypes = [vp, ctypes.c_int, ctypes.c_int64, vp, _i64p, _i32p, _i32p, _i64p, _i64p,
                                       _i64p]
    lib.reshard_plan_slabs.argtypes = [vp, ctypes.c_int64, _i64p, _i64p]
    lib.reshard_plan_status.argtypes = [vp, _i32p, ctypes.c_int]
    lib.reshard_plan_destroy.argtypes = [vp]
    lib.reshard_last_error.argtypes = []
    lib.reshard_last_error.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    return lib


LIB = _load()


def _check(rc: int) -> None:
    if rc != RESHARD_OK:
        raise ReshardError(rc, reshard_last_error())


def reshard_last_error() -> str:
    return LIB.reshard_last_error().decode()


# ------------------------------------------------------------------------ spec containers

@dataclasses.dataclass
class View:
    """Where one rank's shard lives in its buffer: element offset and element strides of the
    local shard (None: dense row-major)."""
    offset: int = 0
    strides: Optional[Sequence[int]] = None


@dataclasses.dataclass
class Spec:
    """One tensor's reshard, as reshard_plan_create takes it: the global shape and dtype
    ("bf16", "f16", "f32", "u8", "i32", "i64"), and on each side the mesh shape and one placement
    per mesh dim ("S<d>" / "R", or torch.distributed.tensor Shard(d) / Replicate()). Optional:
    per-rank views (one per pointer index) and rank permutations (mesh position -> pointer index)."""
    global_shape: Sequence[int]
    dtype: str
    src_mesh: Sequence[int]
    src_placements: Sequence[Any]
    dst_mesh: Sequence[int]
    dst_placements: Sequence[Any]
    src_views: Optional[Sequence[View]] = None
    dst_views: Optional[Sequence[View]] = None
    src_ranks: Optional[Sequence[int]] = None
    dst_ranks: Optional[Sequence[int]] = None


# ------------------------------------------------------------------------- spec marshalling

def _arr(ctype, vals):
    vals = [int(v) for v in vals]
    return (ctype * max(1, len(vals)))(*vals)


def placement_pair(p) -> tuple:
    """(kind, dim) of one placement: "R" / "S<d>", a (kind, dim) pair, or a PyTorch DTensor
    placement object (torch.distributed.tensor.Shard(d) / Replicate())."""
    if isinstance(p, str):
        return (RESHARD_REPLICATE, 0) if p == "R" else (RESHARD_SHARD, int(p[1:]))
    if hasattr(p, "is_shard") and hasattr(p, "is_replicate"):
        if p.is_shard():
            return (RESHARD_SHARD, int(p.dim))
        if p.is_replicate():
            return (RESHARD_REPLICATE, 0)
        raise ReshardError(RESHARD_ERR_UNSUPPORTED, f"placement {p!r} is neither Shard nor Replicate")
    return int(p[0]), int(p[1])


def _placements(pls: Sequence[Any]):
    out = (PlacementT * max(1, len(pls)))()
    for i, p in enumerate(pls):
        out[i].kind, out[i].dim = placement_pair(p)
    return out


def _views(views, capacities, keep):
    if views is None:
        return None
    out = (ViewT * max(1, len(views)))()
    for i, v in enumerate(views):
        out[i].offset_elems = int(getattr(v, "offset", 0))
        st = getattr(v, "strides", None)
        if st is not None:
            a = _arr(ctypes.c_int64, st)
            keep.append(a)
            out[i].strides_elems = a
        out[i].capacity_elems = int(capacities[i]) if capacities is not None else 0
    return out


def make_spec(desc, src_capacity: Optional[Sequence[int]] = None, dst_capacity: Optional[Sequence[int]] = None,
              keep: Optional[list] = None) -> TensorSpecT:
    """Marshal one tensor description into the C struct.

    ``desc`` needs: global_shape, dtype ("bf16", ... or a code), src_mesh, src_placements
    ("R"/"S<d>" or (kind, dim)), dst_mesh, dst_placements; optionally src_views / dst_views
    (objects with .offset and .strides, one per pointer index) and src_ranks / dst_ranks.
    ``keep`` collects the ctypes arrays that must outlive the C call.
    """
    keep = keep if keep is not None else []
    s = TensorSpecT()
    gs = _arr(ctypes.c_int64, desc.global_shape)
    s.ndim = len(desc.global_shape)
    s.global_shape = gs
    s.dtype = DTYPE_CODES[desc.dtype] if isinstance(desc.dtype, str) else int(desc.dtype)
    parts = [gs]
    for side in ("src", "dst"):
        mesh = getattr(desc, f"{side}_mesh")
        ms = _arr(ctypes.c_int64, mesh)
        ranks = getattr(desc, f"{side}_ranks", None)
        rk = _arr(ctypes.c_int32, ranks) if ranks is not None else None
        m = MeshT(len(mesh), ms, rk)
        pl = _placements(getattr(desc, f"{side}_placements"))
        vw = _views(getattr(desc, f"{side}_views", None), src_capacity if side == "src" else dst_capacity, keep)
        setattr(s, f"{side}_mesh", m)
        setattr(s, f"{side}_pl", pl)
        if vw is not None:
            setattr(s, f"{side}_views", vw)
        parts += [ms, rk, pl, vw]
    keep.extend(p for p in parts if p is not None)
    return s


def _spec_dtype():
    """numpy record type laid out exactly like reshard_tensor_spec_t (offsets taken from ctypes)."""
    names, formats, offsets = [], [], []

    def add(name, fmt, off):
        names.append(name)
        formats.append(fmt)
        offsets.append(off)
    add("ndim", "<i4", TensorSpecT.ndim.offset)
    add("global_shape", "<u8", TensorSpecT.global_shape.offset)
    add("dtype", "<i4", TensorSpecT.dtype.offset)
    for side in ("src", "dst"):
        m = getattr(TensorSpecT, f"{side}_mesh").offset
        add(f"{side}_ndim", "<i4", m + MeshT.ndim.offset)
        add(f"{side}_shape", "<u8", m + MeshT.shape.offset)
        add(f"{side}_ranks", "<u8", m + MeshT.ranks.offset)
        add(f"{side}_pl", "<u8", getattr(TensorSpecT, f"{side}_pl").offset)
        add(f"{side}_views", "<u8", getattr(TensorSpecT, f"{side}_views").offset)
    return np.dtype({"names": names, "formats": formats, "offsets": offsets, "itemsize": ctypes.sizeof(TensorSpecT)})


_VIEW_DTYPE = None
_SPEC_DTYPE = None


def pack_specs(descs: Sequence[Any], src_capacity=None, dst_capacity=None):
    """Marshal many tensor descriptions into one contiguous reshard_tensor_spec_t array.

    Every integer goes into a few flat numpy pools (int64: shapes, meshes, strides; int32:
    ranks; placement pairs; view records) and each spec field points into them, so a batch of
    thousands of tensors costs a handful of allocations. Returns (specs, keep): ``specs`` is the
    record array, ``keep`` the pools, which must outlive the C call.
    """
    global _VIEW_DTYPE, _SPEC_DTYPE
    if _SPEC_DTYPE is None:
        _SPEC_DTYPE = _spec_dtype()
        _VIEW_DTYPE = np.dtype({"names": ["offset", "strides", "capacity"], "formats": ["<i8", "<u8", "<i8"],
                                "offsets": [ViewT.offset_elems.offset, ViewT.strides_elems.offset,
                                            ViewT.capacity_elems.offset], "itemsize": ctypes.sizeof(ViewT)})
    n = len(descs)
    i64: List[int] = []
    i32: List[int] = []
    pls: List[int] = []
    views: List[tuple] = []   # (offset, strides index in i64 or -1, capacity)
    rows = []                 # per tensor: field values, pool indices where pointers go
    for t, d in enumerate(descs):
        gs = d.global_shape
        rec = [len(gs), len(i64), DTYPE_CODES[d.dtype] if isinstance(d.dtype, str) else int(d.dtype)]
        i64.extend(int(x) for x in gs)
        for side, caps in (("src", src_capacity), ("dst", dst_capacity)):
            mesh = getattr(d, f"{side}_mesh")
            rec += [len(mesh), len(i64)]
            i64.extend(int(x) for x in mesh)
            ranks = getattr(d, f"{side}_ranks", None)
            if ranks is not None:
                rec.append(len(i32))
                i32.extend(int(x) for x in ranks)
            else:
                rec.append(-1)
            rec.append(len(pls) // 2)
            for p_ in getattr(d, f"{side}_placements"):
                pls += placement_pair(p_)
            vs = getattr(d, f"{side}_views", None)
            if vs is None:
                rec.append(-1)
            else:
                rec.append(len(views))
                cap = caps[t] if caps else None
                for k, v in enumerate(vs):
                    st = getattr(v, "strides", None)
                    si = -1
                    if st is not None:
                        si = len(i64)
                        i64.extend(int(x) for x in st)
                    views.append((int(getattr(v, "offset", 0)), si, int(cap[k]) if cap is not None else 0))
        rows.append(rec)
    pool64 = np.array(i64 or [0], dtype=np.int64)
    pool32 = np.array(i32 or [0], dtype=np.int32)
    poolpl = np.array(pls or [0, 0], dtype=np.int32)
    vrec = np.zeros(max(1, len(views)), dtype=_VIEW_DTYPE)
    b64, b32, bpl, bv = (pool64.ctypes.data, pool32.ctypes.data, poolpl.ctypes.data, vrec.ctypes.data)
    if views:
        va = np.array(views, dtype=np.int64)
        vrec["offset"] = va[:, 0]
        vrec["strides"] = np.where(va[:, 1] >= 0, b64 + 8 * va[:, 1], 0).astype(np.uint64)
        vrec["capacity"] = va[:, 2]
    specs = np.zeros(max(1, n), dtype=_SPEC_DTYPE)
    if n:
        r = np.array(rows, dtype=np.int64)
        specs["ndim"][:n] = r[:, 0]
        specs["global_shape"][:n] = (b64 + 8 * r[:, 1]).astype(np.uint64)
        specs["dtype"][:n] = r[:, 2]
        for k, side in enumerate(("src", "dst")):
            c = 3 + 5 * k
            specs[f"{side}_ndim"][:n] = r[:, c]
            specs[f"{side}_shape"][:n] = (b64 + 8 * r[:, c + 1]).astype(np.uint64)
            specs[f"{side}_ranks"][:n] = np.where(r[:, c + 2] >= 0, b32 + 4 * r[:, c + 2], 0).astype(np.uint64)
            specs[f"{side}_pl"][:n] = (bpl + 8 * r[:, c + 3]).astype(np.uint64)
            specs[f"{side}_views"][:n] = np.where(r[:, c + 4] >= 0, bv + ctypes.sizeof(ViewT) * r[:, c + 4],
                                                  0).astype(np.uint64)
    return specs, [pool64, pool32, poolpl, vrec]


def _spec_ptr(specs):
    return ctypes.cast(ctypes.c_void_p(specs.ctypes.data), ctypes.POINTER(TensorSpecT))


# ------------------------------------------------------------------------------- the calls

class Plan:
    """Owns a reshard_plan_t*; destroyed explicitly or on garbage collection."""

    def __init__(self, handle: int, n_src: int, n_dst: int):
        self.handle = ctypes.c_void_p(handle)
        self.n_src_ptrs = n_src
        self.n_dst_ptrs = n_dst

    def __del__(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            LIB.reshard_plan_destroy(self.handle)
            self.handle = None


def _n_ranks(mesh) -> int:
    n = 1
    for x in mesh:
        n *= int(x)
    return n


def reshard_plan_create(desc, src_capacity=None, dst_capacity=None) -> Plan:
    keep: list = []
    s = make_spec(desc, src_capacity, dst_capacity, keep)
    h = ctypes.c_void_p()
    _check(LIB.reshard_plan_create(ctypes.byref(s), ctypes.byref(h)))
    return Plan(h.value, _n_ranks(desc.src_mesh), _n_ranks(desc.dst_mesh))


def reshard_plan_batch(descs: Sequence[Any], src_capacity=None, dst_capacity=None) -> Plan:
    """One plan over many tensors. Capacities (optional) are per tensor lists of per-rank counts."""
    specs, keep = pack_specs(descs, src_capacity, dst_capacity)
    h = ctypes.c_void_p()
    _check(LIB.reshard_plan_batch(_spec_ptr(specs), len(descs), ctypes.byref(h)))
    del keep
    return Plan(h.value, sum(_n_ranks(d.src_mesh) for d in descs), sum(_n_ranks(d.dst_mesh) for d in descs))


def reshard_plan_blockwise_fp8(descs: Sequence[Any], block=(128, 128), src_capacity=None, dst_capacity=None) -> Plan:
    """FP8 weights (u8) plus their derived blockwise fp32 scales in one plan: weights first,
    then scales, in the pointer arrays too. Capacities (optional) cover the weights only."""
    specs, keep = pack_specs(descs, src_capacity, dst_capacity)
    h = ctypes.c_void_p()
    _check(LIB.reshard_plan_blockwise_fp8(_spec_ptr(specs), len(descs), int(block[0]), int(block[1]), ctypes.byref(h)))
    del keep
    return Plan(h.value, 2 * sum(_n_ranks(d.src_mesh) for d in descs), 2 * sum(_n_ranks(d.dst_mesh) for d in descs))


def _address(p) -> int:
    """A pointer given as an int (0 / None for an empty shard) or as a tensor (its data_ptr())."""
    if p is None:
        return 0
    if hasattr(p, "data_ptr"):
        return int(p.data_ptr())
    return int(p)


def pointer_array(ptrs: Sequence[Any]):
    """Pointers (ints or tensors) as a contiguous uint64 numpy array, passed to the C calls
    without copying.

    Build it once per set of buffers: re-marshalling tens of thousands of pointers per call
    costs milliseconds of host time."""
    import numpy as np
    return np.ascontiguousarray(np.asarray([_address(p) for p in ptrs], dtype=np.uint64))


def _ptrs_arg(ptrs):
    import numpy as np
    if isinstance(ptrs, np.ndarray):
        if ptrs.dtype not in (np.uint64, np.int64) or not ptrs.flags["C_CONTIGUOUS"]:
            raise TypeError("pointer arrays must be contiguous uint64/int64")
        return ptrs.ctypes.data_as(ctypes.POINTER(ctypes.c_void_p)), ptrs
    arr = (ctypes.c_void_p * max(1, len(ptrs)))(*[_address(p) or None for p in ptrs])
    return arr, arr


def reshard_execute(plan: Plan, src_ptrs, dst_ptrs, mode="direct", quant="none", stream: int = 0) -> None:
    """Enqueue the reshard on ``stream`` (a cudaStream_t as int; 0 = legacy default stream).

    ``src_ptrs`` / ``dst_ptrs``: sequences of pointers (ints, or tensors whose data_ptr() is
    used), or uint64 arrays from ``pointer_array`` (no per-call marshalling)."""
    mode = MODES[mode] if isinstance(mode, str) else int(mode)
    quant = QUANTS[quant] if isinstance(quant, str) else int(quant)
    sp, _ks = _ptrs_arg(src_ptrs)
    dp, _kd = _ptrs_arg(dst_ptrs)
    _check(LIB.reshard_execute(plan.handle, sp, dp, mode, quant, ctypes.c_void_p(int(stream) or None)))


def reshard_execute_pack(plan: Plan, src_ptrs, dst_ptrs, send_buf, quant="none", stream: int = 0) -> None:
    """Pack pass with a caller-owned send buffer (``send_buf``: pointer or tensor,
    ``reshard_plan_stats(plan)["message_bytes"]`` bytes). On a partitioned plan it also makes the
    copies whose source and destination are both local; ``dst_ptrs`` may be None otherwise."""
    quant = QUANTS[quant] if isinstance(quant, str) else int(quant)
    sp, _ks = _ptrs_arg(src_ptrs)
    dp, _kd = _ptrs_arg(dst_ptrs) if dst_ptrs is not None else (None, None)
    _check(LIB.reshard_execute_pack(plan.handle, sp, dp, ctypes.c_void_p(_address(send_buf) or None), quant,
                                    ctypes.c_void_p(int(stream) or None)))


def reshard_execute_unpack(plan: Plan, recv_buf, dst_ptrs, quant="none", stream: int = 0) -> None:
    """Unpack pass from a caller-owned receive buffer (``reshard_plan_stats(plan)["recv_bytes"]``)."""
    quant = QUANTS[quant] if isinstance(quant, str) else int(quant)
    dp, _kd = _ptrs_arg(dst_ptrs)
    _check(LIB.reshard_execute_unpack(plan.handle, ctypes.c_void_p(_address(recv_buf) or None), dp, quant,
                                      ctypes.c_void_p(int(stream) or None)))


def reshard_plan_partition(plan: Plan, src_owner: Sequence[int], dst_owner: Sequence[int], world: int, rank: int,
                           striped: bool = True) -> Plan:
    """The share of ``plan`` that process ``rank`` of ``world`` runs; owners map every flat source /
    destination pointer index to the process holding it."""
    so = np.ascontiguousarray(np.asarray(src_owner, dtype=np.int32))
    do = np.ascontiguousarray(np.asarray(dst_owner, dtype=np.int32))
    if so.size != plan.n_src_ptrs or do.size != plan.n_dst_ptrs:
        raise ValueError("one owner per source pointer and per destination pointer")
    h = ctypes.c_void_p()
    _check(LIB.reshard_plan_partition(plan.handle, so.ctypes.data_as(_i32p), do.ctypes.data_as(_i32p), int(world),
                                      int(rank), RESHARD_STRIPED if striped else 0, ctypes.byref(h)))
    return Plan(h.value, plan.n_src_ptrs, plan.n_dst_ptrs)


def reshard_plan_transfers(plan: Plan, phase: int) -> List[Dict[str, int]]:
    """Point-to-point transfers of a partitioned plan's rank in one phase, in posting order."""
    n = ctypes.c_int64()
    _check(LIB.reshard_plan_transfers(plan.handle, int(phase), 0, None, ctypes.byref(n)))
    out = (TransferT * max(1, n.value))()
    _check(LIB.reshard_plan_transfers(plan.handle, int(phase), n.value, out, ctypes.byref(n)))
    return [{f: int(getattr(out[i], f)) for f, _ in TransferT._fields_} for i in range(n.value)]


def reshard_execute_static(plan: Plan, src_ptrs: Sequence[int], dst_ptrs: Sequence[int], stream: int = 0) -> None:
    """Direct-mode reshard that allocates no device memory (descriptor tables go to a fixed
    array inside the library; see include/reshard.h). For callers whose device memory is owned
    elsewhere (an engine's reserved pool, a framework allocator) and must not see cudaMalloc."""
    sp, _ks = _ptrs_arg(src_ptrs)
    dp, _kd = _ptrs_arg(dst_ptrs)
    _check(LIB.reshard_execute_static(plan.handle, sp, dp, ctypes.c_void_p(int(stream) or None)))


def reshard_plan_stats(plan: Plan) -> Dict[str, int]:
    st = StatsT()
    _check(LIB.reshard_plan_stats(plan.handle, ctypes.byref(st)))
    return {f: int(getattr(st, f)) for f in STATS_FIELDS}


def reshard_plan_regions(plan: Plan) -> List[tuple]:
    """[(tensor, src_rank, dst_group, ((lo, hi), ...)), ...] in plan order (global coordinates)."""
    n = ctypes.c_int64()
    _check(LIB.reshard_plan_regions(plan.handle, 0, None, None, None, None, None, ctypes.byref(n)))
    k = n.value
    t = (ctypes.c_int32 * max(1, k))()
    s = (ctypes.c_int32 * max(1, k))()
    g = (ctypes.c_int32 * max(1, k))()
    lo = (ctypes.c_int64 * max(1, k * RESHARD_MAX_DIMS))()
    hi = (ctypes.c_int64 * max(1, k * RESHARD_MAX_DIMS))()
    _check(LIB.reshard_plan_regions(plan.handle, k, t, s, g, lo, hi, ctypes.byref(n)))
    D = RESHARD_MAX_DIMS
    return [(t[i], s[i], g[i], tuple((lo[i * D + d], hi[i * D + d]) for d in range(D))) for i in range(k)]


def reshard_plan_group_members(plan: Plan, g: int) -> List[int]:
    n = ctypes.c_int64()
    _check(LIB.reshard_plan_group_members(plan.handle, g, 0, None, ctypes.byref(n)))
    out = (ctypes.c_int32 * max(1, n.value))()
    _check(LIB.reshard_plan_group_members(plan.handle, g, n.value, out, ctypes.byref(n)))
    return list(out[: n.value])


ITEM_DTYPE = [("src_off", "<i8"), ("dst_off", "<i8"), ("src_pitch", "<i8"), ("dst_pitch", "<i8"),
              ("rows", "<i4"), ("run", "<i4"), ("src", "<i4"), ("group", "<i4"), ("esize", "<i4"),
              ("pad", "<i4", (3,))]


TITEM_DTYPE = [("src_off", "<i8"), ("dst_off", "<i8"), ("src_pitch", "<i8"), ("dst_pitch", "<i8"),
               ("rows", "<i4"), ("cols", "<i4"), ("src", "<i4"), ("group", "<i4"), ("esize", "<i4"),
               ("slab", "<i4"), ("x", "<i4"), ("y", "<i4")]


GITEM_DTYPE = [("src_off", "<i8", (2,)), ("src_pitch", "<i8", (2,)), ("dst_off", "<i8", (2,)),
               ("dst_pitch", "<i8", (2,)), ("run", "<i4", (2,)), ("src", "<i4", (2,)), ("rows", "<i4"),
               ("group", "<i4"), ("esize", "<i4"), ("kind", "<i4")]


def reshard_plan_items(plan: Plan, which: int = 0):
    """(items as a numpy structured array, group_start, member_ptr, member_off) of one table:
    0/1/2 strided-copy items of the direct/pack/unpack pass, 3/4/5 their transposing items, 6/7/8
    their pair items (kind 0: a destination row of two source pieces, direct and unpack passes;
    kind 1: a source row into two message blocks, pack pass; copy items they cover have
    pad[0] == 1)."""
    import numpy as np
    n, ng, nm = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(LIB.reshard_plan_items(plan.handle, which, 0, None, ctypes.byref(n), None, None, None,
                                  ctypes.byref(ng), ctypes.byref(nm)))
    items = np.zeros(n.value, dtype=ITEM_DTYPE if which < 3 else TITEM_DTYPE if which < 6 else GITEM_DTYPE)
    gs = np.zeros(ng.value + 1, np.int32)
    mp = np.zeros(max(1, nm.value), np.int32)
    mo = np.zeros(max(1, nm.value), np.int64)
    _check(LIB.reshard_plan_items(plan.handle, which, n.value, items.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n),
                                  gs.ctypes.data_as(_i32p), mp.ctypes.data_as(_i32p), mo.ctypes.data_as(_i64p),
                                  ctypes.byref(ng), ctypes.byref(nm)))
    return items, gs, mp[: nm.value], mo[: nm.value]


def reshard_plan_slabs(plan: Plan):
    """[(pointer index, esize, base offset, cols, rows, pitch), ...] read by the TMA kernel."""
    n = ctypes.c_int64()
    _check(LIB.reshard_plan_slabs(plan.handle, 0, None, ctypes.byref(n)))
    out = (ctypes.c_int64 * max(1, 6 * n.value))()
    _check(LIB.reshard_plan_slabs(plan.handle, n.value, out, ctypes.byref(n)))
    return [tuple(out[6 * i: 6 * i + 6]) for i in range(n.value)]


def reshard_plan_status(plan: Plan, reset: bool = False) -> int:
    """Device status word of the plan (0 = fine); synchronizes the device."""
    st = ctypes.c_int32()
    _check(LIB.reshard_plan_status(plan.handle, ctypes.byref(st), 1 if reset else 0))
    return int(st.value)


def reshard_plan_destroy(plan: Plan) -> None:
    if plan.handle is not None and plan.handle.value:
        _check(LIB.reshard_plan_destroy(plan.handle))
    plan.handle = None
