"""ctypes loader for the plain-C oracle (TEST INFRASTRUCTURE).

Only tests, smoke() and the bench's CPU-baseline leg may use it. ``build()`` compiles
``oracle.c`` with the host C compiler into ``liboracle.so`` beside it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

from .golden import ESIZE, mesh_coords, shard_box, box_shape

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

ERRORS = {1: "source replicas disagree", 2: "sources leave elements uncovered",
          3: "bad arguments", 4: "out of host memory"}


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(src):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load(path: str):
    """The oracle library at ``path`` with its argument types declared (tests load planted-mistake
    builds of oracle.c this way)."""
    L = ctypes.CDLL(path)
    p64 = ctypes.POINTER(ctypes.c_int64)
    p32 = ctypes.POINTER(ctypes.c_int32)
    pp = ctypes.POINTER(ctypes.c_void_p)
    L.oracle_reshard_tensor.argtypes = [
        ctypes.c_int, p64, ctypes.c_int,
        ctypes.c_int, p64, p32, pp, p64, p64,
        ctypes.c_int, p64, p32, pp, p64, p64,
        ctypes.c_int, pp]
    L.oracle_reshard_tensor.restype = ctypes.c_int
    L.oracle_e4m3.argtypes = [ctypes.c_uint16, ctypes.c_int]
    L.oracle_e4m3.restype = ctypes.c_uint8
    L.oracle_block_exponent.argtypes = [ctypes.POINTER(ctypes.c_uint16)]
    L.oracle_block_exponent.restype = ctypes.c_int
    L.oracle_mxfp8_block.argtypes = [ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_uint8),
                                     ctypes.POINTER(ctypes.c_uint8)]
    L.oracle_mxfp8_block.restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load(_LIB_PATH)
    return _lib


def _i64(v):
    return (ctypes.c_int64 * max(1, len(v)))(*[int(x) for x in v])


def _pl(placements):
    return (ctypes.c_int32 * len(placements))(*[-1 if p == "R" else int(p[1:]) for p in placements])


def _ptrs(arrs):
    return (ctypes.c_void_p * max(1, len(arrs)))(*[a.ctypes.data if a.size else None for a in arrs])


def reshard_tensor(desc, src_bufs: Sequence[np.ndarray], dst_bufs: Sequence[np.ndarray],
                   quant: str = "none", scale_bufs: Optional[Sequence[np.ndarray]] = None, L=None) -> None:
    """Golden reshard of one tensor through the C oracle, in place into byte buffers."""
    L = L or lib()
    nd = len(desc.global_shape)

    def strides(views, mesh, pls):
        if all(v.strides is None for v in views):
            return None
        out = []
        for coord, v in zip(mesh_coords(mesh), views):
            shp = box_shape(shard_box(desc.global_shape, mesh, pls, coord))
            if v.strides is None:
                out.extend(int(np.prod(shp[i + 1:])) for i in range(nd))
            else:
                out.extend(v.strides)
        return _i64(out)

    ss = strides(desc.src_views, desc.src_mesh, desc.src_placements)
    ds = strides(desc.dst_views, desc.dst_mesh, desc.dst_placements)
    rc = L.oracle_reshard_tensor(
        nd, _i64(desc.global_shape), ESIZE[desc.dtype],
        len(desc.src_mesh), _i64(desc.src_mesh), _pl(desc.src_placements), _ptrs(src_bufs),
        _i64([v.offset for v in desc.src_views]), ss,
        len(desc.dst_mesh), _i64(desc.dst_mesh), _pl(desc.dst_placements), _ptrs(dst_bufs),
        _i64([v.offset for v in desc.dst_views]), ds,
        1 if quant == "mxfp8" else 0, _ptrs(scale_bufs) if scale_bufs is not None else None)
    if rc:
        raise RuntimeError(f"C oracle: {desc.name}: {ERRORS.get(rc, rc)}")


def run_workload(wl, src_slab: np.ndarray, src_off, dst_slab: np.ndarray, dst_off,
                 scale_slab: Optional[np.ndarray] = None, scale_off=None, tensors=None, L=None) -> None:
    """Golden reshard of (a subset of) a workload's tensors, in place on host slabs."""
    for ti in (range(len(wl.tensors)) if tensors is None else tensors):
        t = wl.tensors[ti]
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
        reshard_tensor(t, sb, db, wl.quant, cb, L)


def e4m3(bits: int, x: int) -> int:
    return int(lib().oracle_e4m3(bits, x))


def mxfp8_block(bits32: Sequence[int]):
    L = lib()
    arr = (ctypes.c_uint16 * 32)(*bits32)
    out = (ctypes.c_uint8 * 32)()
    sc = ctypes.c_uint8()
    L.oracle_mxfp8_block(arr, out, ctypes.byref(sc))
    return list(out), int(sc.value)
