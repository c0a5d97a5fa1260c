"""Shared test helpers: run a workload through the C ABI on the GPU and compare with the oracle."""
from __future__ import annotations

import itertools
import os

import numpy as np
import torch

import dtensor_resharding_gb300 as R
import synthetic as S
from oracle import coracle, golden as G


def run_gpu(wl, mode="direct", misalign=0, plan=None, execute=True):
    """Allocate, fill sources and canary, plan and execute on cuda. Returns (layout, plan)."""
    lay = S.allocate(wl, "cuda", misalign=misalign)
    S.fill_sources(wl, lay)
    S.fill_canary(lay)
    plan = plan or R.plan_workload(wl)
    if execute:
        sp, dp = R.workload_pointers(wl, lay)
        R.reshard_execute(plan, sp, dp, mode=mode, quant=wl.quant, stream=torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        # no TMA wait timed out and no item reached the aligned walker unaligned
        assert R.reshard_plan_status(plan) == 0
    return lay, plan


def oracle_expected(wl, lay):
    """Host expectation of the whole destination (and scale) slab: canary outside the views."""
    src = lay.src_slab.cpu().numpy()
    want = np.full(lay.dst_slab.numel(), 0xA5, np.uint8)
    wsc = np.full(lay.scale_slab.numel(), 0xA5, np.uint8) if lay.scale_slab is not None else None
    coracle.run_workload(wl, src, lay.src_off, want, lay.dst_off, wsc, lay.scale_off)
    return want, wsc


def assert_matches_oracle(wl, lay):
    want, wsc = oracle_expected(wl, lay)
    got = lay.dst_slab.cpu().numpy()
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{wl.name}: {bad.size} destination bytes differ, first at {bad[:8]}"
    if wsc is not None:
        gs = lay.scale_slab.cpu().numpy()
        bad = np.nonzero(gs != wsc)[0]
        assert bad.size == 0, f"{wl.name}: {bad.size} scale bytes differ, first at {bad[:8]}"


def _mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 16 << 30


def whole_check(wl, lay, workers=None):
    """Whole-output parity at any size, streamed so that host memory stays bounded.

    Tensors are grouped so that no destination buffer is shared between groups; for each group
    the source buffers it reads are copied to the host, the C oracle writes the group's
    destination (and scale) buffers into canary-filled host buffers, and every byte of those
    buffers is compared with the device's (views and the gaps between them). Groups run on a
    thread pool (the oracle and the copies release the GIL). Returns the bytes compared."""
    import concurrent.futures as cf
    es = {k: v[1] for k, v in S.DTYPES.items()}
    quant = wl.quant == "mxfp8"
    n_t = len(wl.tensors)
    parent = list(range(n_t))

    def find(x):
        while parent[x] != x:
            parent[x] = parent[parent[x]]
            x = parent[x]
        return x
    first = {}
    for ti, t in enumerate(wl.tensors):
        for v in t.dst_views:
            if v.buffer in first:
                parent[find(ti)] = find(first[v.buffer])
            else:
                first[v.buffer] = ti
    comps = {}
    for ti in range(n_t):
        comps.setdefault(find(ti), []).append(ti)
    comps = list(comps.values())

    def sbytes(b):
        return wl.src_buffer_numel[b] * es[wl.src_buffer_dtype[b]]

    def dbytes(b):
        return wl.dst_buffer_numel[b] * (1 if quant else es[wl.dst_buffer_dtype[b]])

    def need(tids):
        sb = {v.buffer for ti in tids for v in wl.tensors[ti].src_views}
        db = {v.buffer for ti in tids for v in wl.tensors[ti].dst_views}
        glob = sum(int(np.prod(wl.tensors[ti].global_shape)) * es[wl.tensors[ti].dtype] for ti in tids)
        return sum(sbytes(b) for b in sb) + 2 * sum(dbytes(b) for b in db) + 2 * glob
    est = max(need(c) for c in comps) if comps else 1
    cores = os.cpu_count() or 1
    if workers is None:
        workers = max(1, min(cores, int(0.5 * _mem_available() // max(est, 1))))

    def compact(bufs, size_of):
        off, cur = [0] * (max(bufs) + 1 if bufs else 1), 0
        for b in bufs:
            off[b] = cur
            cur += (size_of(b) + 15) // 16 * 16
        return off, cur

    def one(tids):
        sb = sorted({v.buffer for ti in tids for v in wl.tensors[ti].src_views})
        db = sorted({v.buffer for ti in tids for v in wl.tensors[ti].dst_views})
        s_off, s_n = compact(sb, sbytes)
        d_off, d_n = compact(db, dbytes)
        src = np.empty(max(1, s_n), np.uint8)
        for b in sb:
            torch.from_numpy(src[s_off[b]: s_off[b] + sbytes(b)]).copy_(lay.src_slab[lay.src_off[b]: lay.src_off[b] + sbytes(b)])
        want = np.full(max(1, d_n), 0xA5, np.uint8)
        got = np.empty(max(1, d_n), np.uint8)
        wsc = gsc = c_off = None
        if quant:
            c_off, c_n = compact(db, lambda b: wl.dst_buffer_numel[b] // 32)
            wsc = np.full(max(1, c_n), 0xA5, np.uint8)
            gsc = np.empty(max(1, c_n), np.uint8)
        coracle.run_workload(wl, src, s_off, want, d_off, wsc, c_off, tensors=tids)
        n = 0
        for b in db:
            nb = dbytes(b)
            torch.from_numpy(got[d_off[b]: d_off[b] + nb]).copy_(lay.dst_slab[lay.dst_off[b]: lay.dst_off[b] + nb])
            bad = np.count_nonzero(got[d_off[b]: d_off[b] + nb] != want[d_off[b]: d_off[b] + nb])
            assert bad == 0, f"{wl.name}: destination buffer {b}: {bad} bytes differ from the oracle"
            n += nb
            if quant:
                nc = wl.dst_buffer_numel[b] // 32
                torch.from_numpy(gsc[c_off[b]: c_off[b] + nc]).copy_(
                    lay.scale_slab[lay.scale_off[b]: lay.scale_off[b] + nc])
                bad = np.count_nonzero(gsc[c_off[b]: c_off[b] + nc] != wsc[c_off[b]: c_off[b] + nc])
                assert bad == 0, f"{wl.name}: scale buffer {b}: {bad} bytes differ from the oracle"
                n += nc
        return n

    if lay.dst_slab.is_cuda:
        torch.cuda.synchronize()
    with cf.ThreadPoolExecutor(workers) as ex:
        return sum(ex.map(one, comps))


def _gather(slab: torch.Tensor, offsets: np.ndarray, nbytes: int) -> np.ndarray:
    idx = torch.from_numpy((offsets[:, None] + np.arange(nbytes)[None, :]).reshape(-1)).to(slab.device)
    return slab[idx].cpu().numpy().reshape(len(offsets), nbytes)


def _dst_shape(t, r):
    return G.box_shape(G.shard_box(t.global_shape, t.dst_mesh, t.dst_placements, G.mesh_coords(t.dst_mesh)[r]))


def _src_shape(t, s):
    return G.box_shape(G.shard_box(t.global_shape, t.src_mesh, t.src_placements, G.mesh_coords(t.src_mesh)[s]))


def sampled_check(wl, lay, per_tensor=8, seed=0, max_tensors=None, corners=False):
    """Sampled parity at full size: the oracle maps each sampled destination element to the
    source element that must supply it; the bytes must be equal (copy workloads). With
    ``corners`` the first and last element of every destination shard are sampled too."""
    rng = np.random.Generator(np.random.PCG64(seed))
    tids = range(len(wl.tensors))
    if max_tensors and len(wl.tensors) > max_tensors:
        tids = sorted(rng.choice(len(wl.tensors), size=max_tensors, replace=False))
    src_off, dst_off, es_list = [], [], []
    for ti in tids:
        t = wl.tensors[ti]
        es = G.ESIZE[t.dtype]
        picks = []
        for _ in range(per_tensor):
            r = int(rng.integers(0, t.n_dst))
            shp = _dst_shape(t, r)
            if int(np.prod(shp)) == 0:
                continue
            picks.append((r, shp, tuple(int(rng.integers(0, n)) for n in shp)))
        if corners:
            for r in range(t.n_dst):
                shp = _dst_shape(t, r)
                if int(np.prod(shp)) > 0:
                    picks += [(r, shp, tuple(0 for _ in shp)), (r, shp, tuple(n - 1 for n in shp))]
        for r, shp, idx in picks:
            s, sidx = G.dst_element_source(t, r, idx)
            sv, dv = t.src_views[s], t.dst_views[r]
            src_off.append(lay.src_off[sv.buffer] + es * G.element_offset(sv, _src_shape(t, s), sidx))
            dst_off.append(lay.dst_off[dv.buffer] + es * G.element_offset(dv, shp, idx))
            es_list.append(es)
    n = 0
    for es in sorted(set(es_list)):
        sel = [i for i, e in enumerate(es_list) if e == es]
        a = _gather(lay.src_slab, np.array([src_off[i] for i in sel], np.int64), es)
        b = _gather(lay.dst_slab, np.array([dst_off[i] for i in sel], np.int64), es)
        bad = np.nonzero((a != b).any(axis=1))[0]
        assert bad.size == 0, f"{wl.name}: {bad.size} of {len(a)} sampled {es}-byte elements differ"
        n += len(a)
    return n


def sampled_check_mxfp8(wl, lay, per_tensor=8, seed=0):
    """Sampled parity of MXFP8 blocks: the oracle gathers the block's 32 source elements one by
    one and quantizes them; the 32 E4M3 bytes and the E8M0 byte must be equal."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = 0
    for t in wl.tensors:
        for _ in range(per_tensor):
            r = int(rng.integers(0, t.n_dst))
            shp = _dst_shape(t, r)
            outer = tuple(int(rng.integers(0, x)) for x in shp[:-1])
            b = int(rng.integers(0, shp[-1] // 32))
            offs = []
            for i in range(32):
                idx = outer + (32 * b + i,)
                s, sidx = G.dst_element_source(t, r, idx)
                sv = t.src_views[s]
                offs.append(lay.src_off[sv.buffer] + 2 * G.element_offset(sv, _src_shape(t, s), sidx))
            vals = _gather(lay.src_slab, np.array(offs, np.int64), 2)
            bits = [int(v[0]) | (int(v[1]) << 8) for v in vals]
            codes, scale = coracle.mxfp8_block(bits)
            dv = t.dst_views[r]
            e0 = G.element_offset(dv, shp, outer + (32 * b,))
            got = _gather(lay.dst_slab, np.array([lay.dst_off[dv.buffer] + e0], np.int64), 32)[0]
            gs = _gather(lay.scale_slab, np.array([lay.scale_off[dv.buffer] + e0 // 32], np.int64), 1)[0, 0]
            assert list(got) == codes and int(gs) == scale, (t.name, r, outer, b)
            n += 1
    return n


def round_trip_desc(t):
    return S.TensorDesc(t.name + ".back", t.global_shape, t.dtype, t.dst_mesh, t.dst_placements,
                        t.src_mesh, t.src_placements, t.dst_views, t.src_views, t.seed, t.std)


def free(*objs):
    for o in objs:
        del o
    torch.cuda.empty_cache()
