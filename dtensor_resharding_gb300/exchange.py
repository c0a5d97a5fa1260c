"""Multi-process reshard: pack, exchange the messages, unpack.

The Reshard collective moves each process's source regions to the processes that hold their
destinations (news article on NVIDIA's Reshard collective, "The Reshard collective" and "How
NCCL M2N Reshard maximizes network bandwidth"; NeMo-RL design doc "NCCL Reshard Refit
(Experimental)", "xferdtensor Transports": batched point-to-point transfers, receives striped
across destination replicas and then spread inside each replica group). Here every process runs
its share of a plan (``reshard_plan_partition``):

1. ``reshard_execute_pack`` copies the regions whose source and destination are both local and
   packs the outgoing messages into the send buffer (kernels on the given stream);
2. the transfers of phase 1, then of phase 2 (``reshard_plan_transfers``) move message bytes
   between processes through ``torch.distributed`` point-to-point operations, posted as one
   batch per phase (one NCCL group on GPUs; gloo on CPU tensors);
3. ``reshard_execute_unpack`` writes the received messages into the local destinations
   (quantizing to MXFP8 when asked).

This module only posts the library's transfer lists; every byte of the data path on a GPU is
moved by the library's kernels or by the communication library. ``loopback_transfers`` plays
the transfers of several ranks inside one process with device copies, so that the whole path
can be checked on one GPU.
"""
from __future__ import annotations

from typing import Optional, Sequence

from . import binding as B


def _bufs(plan, send_buf, recv_buf):
    st = B.reshard_plan_stats(plan)
    for name, buf, need in (("send_buf", send_buf, st["message_bytes"]), ("recv_buf", recv_buf, st["recv_bytes"])):
        if need and (buf is None or buf.numel() * buf.element_size() < need):
            raise ValueError(f"{name} must hold {need} bytes")
    return st


def _flat(buf):
    import torch
    return buf.view(-1).view(torch.uint8)


_started = {}  # process groups that have run a collective with every rank (id -> the group)


def run_transfers(plan, send_buf, recv_buf, group=None) -> None:
    """Post this rank's transfers of phase 1, wait for them, then those of phase 2.

    ``send_buf`` / ``recv_buf``: contiguous tensors (uint8 views are taken) on the device the
    process group communicates from. Peers are ranks of ``group`` (the default group if None).
    A rank with nothing to send or receive in a phase posts nothing; since a batched
    point-to-point call that is a group's first collective must include every rank (NCCL), the
    first call on a group starts with a barrier of the whole group."""
    import torch.distributed as dist
    _bufs(plan, send_buf, recv_buf)
    g = group if group is not None else dist.distributed_c10d._get_default_group()
    if _started.get(id(g)) is not g:
        dist.barrier(group=group)
        _started[id(g)] = g  # held, so that its id is not reused by a later group
    sb = _flat(send_buf) if send_buf is not None else None
    rb = _flat(recv_buf) if recv_buf is not None else None
    for phase in (1, 2):
        ops = []
        for t in B.reshard_plan_transfers(plan, phase):
            buf = sb if t["buf"] == B.RESHARD_SEND_BUF else rb
            view = buf[t["offset"]: t["offset"] + t["bytes"]]
            peer = t["peer"] if group is None else dist.get_global_rank(group, t["peer"])
            op = dist.isend if t["dir"] == B.RESHARD_SEND else dist.irecv
            ops.append(dist.P2POp(op, view, peer, group))
        if ops:
            for work in dist.batch_isend_irecv(ops):
                work.wait()


def reshard_exchange(plan, src_ptrs, dst_ptrs, send_buf, recv_buf, quant="none", group=None,
                     stream: Optional[int] = None) -> None:
    """One rank's whole reshard: pack, both transfer phases, unpack.

    ``plan`` is this rank's partitioned plan; pointer arrays are global (other ranks' entries
    may be 0). Packing and unpacking run on ``stream`` (default: the current CUDA stream); the
    communication library orders its transfers after the work already on the current stream."""
    import torch
    st = _bufs(plan, send_buf, recv_buf)
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else 0
    B.reshard_execute_pack(plan, src_ptrs, dst_ptrs, send_buf if st["message_bytes"] else None, quant, stream)
    run_transfers(plan, send_buf, recv_buf, group)
    B.reshard_execute_unpack(plan, recv_buf if st["recv_bytes"] else None, dst_ptrs, quant, stream)


def loopback_transfers(plans: Sequence, send_bufs: Sequence, recv_bufs: Sequence) -> int:
    """Play every transfer of ranks 0..len(plans)-1 inside one process: in each phase, rank a's
    k-th send to rank b is copied into rank b's k-th receive from rank a (the in-order matching
    of point-to-point transfers). Returns the bytes copied. Used to check the multi-rank path on
    one device; buffers are tensors (any device)."""
    moved = 0
    for phase in (1, 2):
        sends, recvs = {}, {}
        for r, p in enumerate(plans):
            for t in B.reshard_plan_transfers(p, phase):
                key = (r, t["peer"]) if t["dir"] == B.RESHARD_SEND else (t["peer"], r)
                (sends if t["dir"] == B.RESHARD_SEND else recvs).setdefault(key, []).append(t)
        if set(sends) != set(recvs):
            raise RuntimeError(f"phase {phase}: unmatched transfer pairs {set(sends) ^ set(recvs)}")
        for (a, b), ss in sends.items():
            rr = recvs[(a, b)]
            if len(ss) != len(rr):
                raise RuntimeError(f"phase {phase}: {len(ss)} sends from {a} to {b} against {len(rr)} receives")
            for s, r in zip(ss, rr):
                if s["bytes"] != r["bytes"]:
                    raise RuntimeError(f"phase {phase}: transfer sizes differ between {a} and {b}")
                src = _flat(send_bufs[a] if s["buf"] == B.RESHARD_SEND_BUF else recv_bufs[a])
                dst = _flat(recv_bufs[b])
                dst[r["offset"]: r["offset"] + r["bytes"]].copy_(src[s["offset"]: s["offset"] + s["bytes"]])
                moved += s["bytes"]
    return moved
