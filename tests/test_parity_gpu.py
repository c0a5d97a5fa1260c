"""GPU parity: the CUDA path through the C ABI against the oracle, byte for byte (tolerance 0).

Small cases (whole slabs compared with the C oracle, canary bytes included) span several
work items, ragged tails, uneven and empty chunks, misaligned buffers, both modes and MXFP8.
The full-size workloads of the five headline configurations are compared whole as well
(streamed tensor group by tensor group through the C oracle, every destination and scale byte,
tolerance 0), after a fast sampled pre-check that the oracle computes element by element; the
other full-size workloads are checked on samples and by the A -> B -> A round trip, which must
give the sources back unchanged.
"""
import numpy as np
import pytest
import torch

import synthetic as S

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import dtensor_resharding_gb300 as R
    from harness import (assert_matches_oracle, run_gpu, sampled_check, sampled_check_mxfp8,
                         round_trip_desc, whole_check)

SMALL = {
    "example_8x8": lambda: S.example_8x8(),
    "dense_ragged": lambda: S.dense_ffn(layers=2, hidden=256, ffn=1000),
    "dense_interleaved_fused": lambda: S.dense_ffn(layers=1, hidden=320, ffn=1096, fused="interleave"),
    "dense_unfused_tp8_to_dp4tp2": lambda: S.dense_ffn(layers=1, hidden=128, ffn=2048, fused="none",
                                                      dp_dst=4, tp_dst=2),
    "moe_ep16_to_ep8": lambda: S.moe_experts(layers=1, experts=32, hidden=256, ffn=96, dst="ep8"),
    "uneven_tp6_to_tp5": lambda: S.uneven_tp(rows=1433, cols=409),
    "mesh2x4_to_3": lambda: S.mesh2d_to_1d(rows=1434, cols=4096, variant="1d"),
    "mesh2x4_to_3x2": lambda: S.mesh2d_to_1d(rows=143, cols=409, variant="2d"),
    "many_small": lambda: S.many_small(n=150),
    "long_run_f32": lambda: S.uneven_tp(rows=3000, cols=1000, src=3, dst=7, dtype="f32"),
    "u8_odd": lambda: S.mesh2d_to_1d(rows=77, cols=333, variant="2d", dtype="u8"),
    "transpose_dst_bf16": lambda: S.transposed(shape=(300, 200), src_mesh=(4,), src_pl=("S0",)),
    "transpose_dst_bf16_big_tiles": lambda: S.transposed(shape=(1100, 640), src_mesh=(2,), src_pl=("S1",),
                                                         dst_mesh=(3,), dst_pl=("S0",)),
    "transpose_src_f32": lambda: S.transposed(shape=(130, 257), src_mesh=(3,), src_pl=("S1",), dst_mesh=(2,),
                                              dst_pl=("S0",), side="src", dtype="f32"),
    "transpose_both_u8": lambda: S.transposed(shape=(77, 300), src_mesh=(2,), src_pl=("S0",), dst_mesh=(2, 2),
                                              dst_pl=("S1", "R"), side="both", dtype="u8"),
    "transpose_3d_i64": lambda: S.transposed(shape=(3, 70, 90), src_mesh=(3,), src_pl=("S0",), dst_mesh=(2,),
                                             dst_pl=("S2",), dtype="i64"),
    "qkv_kv_below_tp_8_to_8": lambda: S.qkv_kv_below_tp(layers=1, q_heads=16, kv_heads=2, head_dim=16, hidden=96),
    "qkv_kv_below_tp_8_to_4": lambda: S.qkv_kv_below_tp(layers=2, q_heads=16, kv_heads=2, head_dim=16, hidden=96,
                                                        tp_dst=4),
    "qkv_kv_below_tp_4_to_8": lambda: S.qkv_kv_below_tp(layers=1, q_heads=16, kv_heads=2, head_dim=24, hidden=80,
                                                        tp_src=4, tp_dst=8),
    "moe_w13_per_expert": lambda: S.moe_w13(layers=1, experts=8, hidden=96, ffn=64, tp_dst=4, per_expert_src=True),
    "moe_w13_stacked_ep4": lambda: S.moe_w13(layers=1, experts=8, hidden=96, ffn=64, ep_src=4, tp_dst=4,
                                             per_expert_src=False),
    "moe_fp8_blockwise": lambda: S.moe_fp8_blockwise(layers=1, experts=4, hidden=256, ffn=384, ep_src=2, dp_src=2,
                                                     tp_dst=3, dp_dst=2),
    "identity_tp4": lambda: _one((1000, 333), (4,), ("S0",), (4,), ("S0",)),
    "broadcast_16_replicas": lambda: _one((100, 300), (1,), ("R",), (16,), ("R",)),
    "nearly_empty_1x1": lambda: _one((1, 1), (2,), ("S0",), (3,), ("S1",)),
    "replicated_source_to_2d": lambda: _one((257, 130), (3, 2), ("R", "S1"), (2, 2), ("S0", "S1")),
    "aligned_rows_with_byte_tails": lambda: _padded((64, 1000), 1024, 504),
    "transpose_mixed_bf16_f32_one_plan": lambda: _merge(
        S.transposed(shape=(300, 200), src_mesh=(4,), src_pl=("S0",)),
        S.transposed(shape=(130, 257), src_mesh=(3,), src_pl=("S1",), dst_mesh=(2,), dst_pl=("S0",),
                     dtype="f32", seed=7)),
    "run_shorter_than_a_word": lambda: _one((1, 3), (1,), ("R",), (2,), ("R",)),
}


def _merge(a, b):
    """One workload holding both workloads' tensors (b's buffers renumbered after a's)."""
    import dataclasses
    ns, nd = len(a.src_buffer_numel), len(a.dst_buffer_numel)
    tb = []
    for t in b.tensors:
        tb.append(dataclasses.replace(
            t, src_views=[dataclasses.replace(v, buffer=v.buffer + ns) for v in t.src_views],
            dst_views=[dataclasses.replace(v, buffer=v.buffer + nd) for v in t.dst_views]))
    return S.Workload(a.name + "+" + b.name, a.tensors + tb, src_buffer_numel=a.src_buffer_numel + b.src_buffer_numel,
                      src_buffer_dtype=a.src_buffer_dtype + b.src_buffer_dtype,
                      dst_buffer_numel=a.dst_buffer_numel + b.dst_buffer_numel,
                      dst_buffer_dtype=a.dst_buffer_dtype + b.dst_buffer_dtype)


def _padded(shape, src_pitch, dst_pitch):
    """One replica into a 2-way column split, both sides with padded row pitches that keep every
    row start 16-byte aligned while the runs (1000 bytes) end 8 bytes into a word."""
    t = S.TensorDesc("w", shape, "bf16", (1,), ("R",), (2,), ("S1",), [S.View(0, 0, (src_pitch, 1))],
                     [S.View(0, 0, (dst_pitch, 1)), S.View(1, 0, (dst_pitch, 1))], seed=37)
    return S.workloads._size_buffers(S.Workload("padded", [t]), 1, 2)


def _one(shape, sm, sp, dm, dp, dtype="bf16", quant="none"):
    import numpy as _np
    ns, nd = int(_np.prod(sm)), int(_np.prod(dm))
    t = S.TensorDesc("w", shape, dtype, sm, sp, dm, dp, [S.View(i) for i in range(ns)], [S.View(i) for i in range(nd)],
                     seed=31)
    return S.workloads._size_buffers(S.Workload("one", [t], quant=quant), ns, nd)


def _as_i16(x):
    """int32 bit patterns in [0, 65536) or [-32768, 32768) -> int16 with the same low 16 bits."""
    x = x & 0xFFFF
    return torch.where(x >= 32768, x - 65536, x).to(torch.int16)


@pytest.fixture(autouse=True)
def _cleanup():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["direct", "packed"])
@pytest.mark.parametrize("misalign", [0, 2, 6])
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workloads_bit_exact(name, misalign, mode):
    wl = SMALL[name]()
    if any(misalign % S.DTYPES[t.dtype][1] for t in wl.tensors):
        pytest.skip("buffer offset must be a multiple of the element size")
    lay, plan = run_gpu(wl, mode=mode, misalign=misalign)
    assert_matches_oracle(wl, lay)


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_transposed_layouts_use_tma_and_report_no_timeouts(mode):
    """Transposed shards go through the TMA kernel (aligned slabs) or its plain-load fallback
    (unaligned buffers); both must match the oracle and leave the status word clear."""
    for misalign in (0, 2):
        wl = S.transposed(shape=(1100, 640), src_mesh=(2,), src_pl=("S1",), dst_mesh=(3,), dst_pl=("S0",))
        lay, plan = run_gpu(wl, mode=mode, misalign=misalign)
        assert_matches_oracle(wl, lay)
        assert R.reshard_plan_status(plan) == 0
        assert len(R.reshard_plan_items(plan, 3)[0]) > 0


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_brute_force_small_meshes(mode):
    """Random meshes (<= 3 dims, <= 4 each), every placement kind, element-id payloads."""
    for wl in S.brute_force_cases(80, seed=21):
        lay, plan = run_gpu(wl, mode=mode)
        assert_matches_oracle(wl, lay)


@pytest.mark.parametrize("mode", ["direct", "packed"])
@pytest.mark.parametrize("misalign", [0, 4])
def test_mxfp8_small_bit_exact(mode, misalign):
    wl = S.moe_experts(layers=1, experts=16, hidden=256, ffn=256, dst="tp4")
    lay, plan = run_gpu(wl, mode=mode, misalign=misalign)
    assert_matches_oracle(wl, lay)


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_mxfp8_six_replicas(mode):
    """A quantized destination replicated 6 ways: more replicas than one quantizer pass holds."""
    wl = _one((64, 128), (2,), ("S0",), (6, 2), ("R", "S1"), quant="mxfp8")
    lay, plan = run_gpu(wl, mode=mode)
    assert_matches_oracle(wl, lay)


def test_mxfp8_special_values_bit_exact():
    """Zero blocks, -0, Inf/NaN blocks, subnormals, saturation and midpoints through the kernel."""
    wl = S.moe_experts(layers=1, experts=8, hidden=64, ffn=128, ep_src=4, dst="tp4")
    lay, plan = run_gpu(wl, execute=False)
    src = lay.src_slab.view(torch.int16)
    n = src.numel()
    g = torch.Generator(device="cuda").manual_seed(5)
    special = torch.tensor([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC1, 0x0001, 0x8001, 0x007F, 0x43E0, 0x43F0,
                            0x4400, 0x3F88, 0xBF88, 0x7F7F, 0xFF7F, 0x3A80], dtype=torch.int32, device="cuda")
    pick = torch.randint(0, special.numel(), (n,), generator=g, device="cuda")
    rand = torch.randint(-32768, 32767, (n,), generator=g, device="cuda", dtype=torch.int32)
    mixed = torch.where(torch.rand(n, generator=g, device="cuda") < 0.3, special[pick], rand)
    # some blocks entirely zero
    mixed = mixed.view(-1, 32)
    mixed[::7] = 0
    src.copy_(_as_i16(mixed.view(-1)))
    # replicas of a source do not exist here (EP sources are disjoint), so any bits are valid input
    sp, dp = R.workload_pointers(wl, lay)
    R.reshard_execute(plan, sp, dp, quant="mxfp8")
    torch.cuda.synchronize()
    assert_matches_oracle(wl, lay)


def test_mxfp8_every_bf16_pattern_at_many_scales():
    """All 65,536 BF16 patterns through the kernel's conversion under many block scales: each
    block holds one scale-setting element and 31 patterns; compared with the C oracle."""
    wl = S.moe_experts(layers=1, experts=4, hidden=64, ffn=2048, ep_src=4, dst="tp4")
    lay, plan = run_gpu(wl, execute=False)
    src = lay.src_slab.view(torch.int16)
    pats = torch.arange(65536, dtype=torch.int32, device="cuda")
    finite = pats[(pats & 0x7F80) != 0x7F80]
    blocks = src.numel() // 32
    body = finite.repeat((blocks * 31) // finite.numel() + 1)[: blocks * 31].view(blocks, 31)
    # leading element sets amax: exponents spread over the whole BF16 range
    lead = ((torch.arange(blocks, device="cuda", dtype=torch.int32) % 254) + 1) << 7
    x = torch.cat([lead[:, None], body], dim=1)
    src.copy_(_as_i16(x.view(-1)))
    sp, dp = R.workload_pointers(wl, lay)
    R.reshard_execute(plan, sp, dp, quant="mxfp8")
    torch.cuda.synchronize()
    assert_matches_oracle(wl, lay)


def test_execute_twice_and_pointer_change():
    """Re-executing a plan with new buffers re-uploads the pointer table."""
    wl = S.dense_ffn(layers=1, hidden=128, ffn=512)
    lay1, plan = run_gpu(wl)
    assert_matches_oracle(wl, lay1)
    lay2, _ = run_gpu(wl, plan=plan, misalign=2)
    assert_matches_oracle(wl, lay2)
    lay3, _ = run_gpu(wl, plan=plan, mode="packed")
    assert_matches_oracle(wl, lay3)


def test_streams_are_honoured():
    wl = S.dense_ffn(layers=1, hidden=256, ffn=1024)
    lay, plan = run_gpu(wl, execute=False)
    s = torch.cuda.Stream()
    sp, dp = R.workload_pointers(wl, lay)
    with torch.cuda.stream(s):
        R.reshard_execute(plan, sp, dp, stream=s.cuda_stream)
    s.synchronize()
    assert_matches_oracle(wl, lay)


# ------------------------------------------------------------------ full sizes, sampled

def _full(wl_fn, mode, sampler, **kw):
    wl = wl_fn()
    lay, plan = run_gpu(wl, mode=mode)
    n = sampler(wl, lay, **kw)
    assert n > 0
    return wl, lay, plan


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_full_dense_ffn_whole_and_round_trip(mode):
    wl, lay, plan = _full(S.dense_ffn, mode, sampled_check, per_tensor=64, corners=True)
    assert whole_check(wl, lay) == wl.dst_bytes()
    # A -> B -> A: the destinations resharded back reproduce the (fused) sources exactly
    back = S.Workload(wl.name + ".back", [round_trip_desc(t) for t in wl.tensors],
                      src_buffer_numel=wl.dst_buffer_numel, src_buffer_dtype=wl.dst_buffer_dtype,
                      dst_buffer_numel=wl.src_buffer_numel, dst_buffer_dtype=wl.src_buffer_dtype)
    bplan = R.plan_workload(back)
    out = torch.empty_like(lay.src_slab)
    out.copy_(lay.src_slab)
    lay.src_slab.fill_(0x5A)
    flip = S.Layout(lay.dst_slab, lay.src_slab, None, lay.dst_off, lay.src_off, None)
    sp, dp = R.workload_pointers(back, flip)
    R.reshard_execute(bplan, sp, dp, mode=mode)
    torch.cuda.synchronize()
    for b, (off, n) in enumerate(zip(lay.src_off, wl.src_buffer_numel)):
        nb = n * S.DTYPES[wl.src_buffer_dtype[b]][1]
        assert torch.equal(lay.src_slab[off: off + nb], out[off: off + nb]), f"source buffer {b} changed"


def test_full_moe_ep16_to_ep8_whole():
    wl, lay, _ = _full(lambda: S.moe_experts(dst="ep8"), "direct", sampled_check, per_tensor=64, corners=True)
    assert whole_check(wl, lay) == wl.dst_bytes()


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_full_moe_tp4_mxfp8_whole(mode):
    wl, lay, _ = _full(lambda: S.moe_experts(dst="tp4"), mode, sampled_check_mxfp8, per_tensor=6)
    assert whole_check(wl, lay) == wl.dst_bytes()


def test_full_edge_mix_bit_exact():
    for wl in (S.uneven_tp(), S.mesh2d_to_1d(variant="1d"), S.mesh2d_to_1d(variant="2d")):
        for mode in ("direct", "packed"):
            lay, plan = run_gpu(wl, mode=mode)
            assert_matches_oracle(wl, lay)


@pytest.mark.parametrize("name", ["qkv_32x64q2kv128x8192_tp8_to_tp4", "moe_w13_48x128x768x2048_ep8_to_tp4",
                                  "moe_w13_4x128x768x2048_per_expert_to_tp4",
                                  "moe_fp8_8x128x768x2048_dp2ep8_to_dp8tp2_b128x128"])
def test_full_next_rows_sampled(name):
    _full(lambda: S.workload_by_name(name), "direct", sampled_check, per_tensor=16, max_tensors=400, corners=True)


def test_full_many_small_whole():
    wl, lay, _ = _full(S.many_small, "direct", sampled_check, per_tensor=4)
    assert whole_check(wl, lay) == wl.dst_bytes()


@pytest.mark.parametrize("side", ["dst", "src"])
@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_full_transposed_destination_sampled(mode, side):
    wl, lay, plan = _full(lambda: S.workload_by_name(f"transpose_32x14336x4096_tp8_to_dp2tp2_{side}_colmajor"), mode,
                          sampled_check, per_tensor=64, corners=True)
    assert R.reshard_plan_status(plan) == 0


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_full_large_offsets_sampled(mode):
    """Buffers of 3.2e9 elements (6.4 GB) on both sides, beyond 32-bit element offsets: copy
    items and TMA tiles far into them, and every shard's first and last element."""
    wl, lay, plan = _full(S.large_offsets, mode, sampled_check, per_tensor=512, corners=True)
    assert R.reshard_plan_status(plan) == 0
    assert max(wl.src_buffer_numel) > 2 ** 31 and max(wl.dst_buffer_numel) > 2 ** 31


@pytest.mark.parametrize("mode", ["direct", "packed"])
def test_fuzzed_layouts_bit_exact(mode):
    """Random shapes, meshes, dtypes and per-rank layouts; copy, funnel-shift and TMA paths."""
    for i, wl in enumerate(S.fuzz_cases(60, seed=23)):
        lay, plan = run_gpu(wl, mode=mode, misalign=[0, 8][i % 2])
        assert_matches_oracle(wl, lay)


@pytest.mark.parametrize("mode", ["direct", "packed"])
@pytest.mark.parametrize("name", ["dense", "mesh_gather", "transposed"])
def test_execute_replays_from_a_cuda_graph(name, mode):
    """Once a plan has run with some pointers, executes with the same pointers only launch
    kernels, so they can be captured into a CUDA graph and replayed: aligned items, gather items
    (direct and unpack passes, their resolved tables already uploaded) and TMA transposes."""
    wl = {"dense": lambda: S.dense_ffn(layers=1, hidden=256, ffn=1024),
          "mesh_gather": lambda: S.mesh2d_to_1d(rows=1434, cols=4096, variant="2d"),
          "transposed": lambda: S.transposed(shape=(300, 256), src_mesh=(4,), src_pl=("S0",))}[name]()
    lay, plan = run_gpu(wl, mode=mode)           # binds the plan and uploads its tables
    S.fill_canary(lay)
    sp, dp = R.workload_pointers(wl, lay)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        R.reshard_execute(plan, sp, dp, mode=mode, stream=s.cuda_stream)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert R.reshard_plan_status(plan) == 0
    assert_matches_oracle(wl, lay)
    if name == "mesh_gather":
        assert R.reshard_plan_stats(plan)["last_gather_items"] > 0


def _pinned_like(t, fill=None):
    h = torch.empty(t.numel(), dtype=t.dtype, pin_memory=True)
    if fill is None:
        h.copy_(t)
    else:
        h.fill_(fill)
    return h


HOST_CASES = {
    "dense": lambda: S.dense_ffn(layers=1, hidden=256, ffn=1000),
    "transposed": lambda: S.transposed(shape=(300, 256), src_mesh=(4,), src_pl=("S0",)),
    "moe_tp4_mxfp8": lambda: S.moe_experts(layers=1, experts=16, hidden=256, ffn=128, dst="tp4"),
    "many_small": lambda: S.many_small(n=20),
    "mesh2x4_to_3x2_gather": lambda: S.mesh2d_to_1d(rows=143, cols=409, variant="2d"),
}


@pytest.mark.parametrize("where", ["host_host", "host_dev", "dev_host"])
@pytest.mark.parametrize("mode", ["direct", "packed"])
@pytest.mark.parametrize("name", sorted(HOST_CASES))
def test_page_locked_host_buffers(name, mode, where):
    """Sources and/or destinations in page-locked host memory: the kernels read and write it in
    place (transposing regions through plain loads, not TMA); bytes equal the oracle's."""
    import dataclasses
    wl = HOST_CASES[name]()
    lay, _ = run_gpu(wl, execute=False, misalign=2 if name == "many_small" else 0)
    kw = {}
    if where in ("host_host", "host_dev"):
        kw["src_slab"] = _pinned_like(lay.src_slab)
    if where in ("host_host", "dev_host"):
        kw["dst_slab"] = _pinned_like(lay.dst_slab, 0xA5)
        if lay.scale_slab is not None:
            kw["scale_slab"] = _pinned_like(lay.scale_slab, 0xA5)
    hl = dataclasses.replace(lay, **kw)
    plan = R.plan_workload(wl)
    sp, dp = R.workload_pointers(wl, hl)
    R.reshard_execute(plan, sp, dp, mode=mode, quant=wl.quant, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert R.reshard_plan_status(plan) == 0
    assert_matches_oracle(wl, hl)


def test_pageable_host_memory_is_refused_before_any_launch():
    wl = S.dense_ffn(layers=1, hidden=256, ffn=1000)
    lay, plan = run_gpu(wl, execute=False)
    pageable = torch.empty(lay.src_slab.numel(), dtype=torch.uint8)   # not page-locked
    import dataclasses
    sp, dp = R.workload_pointers(wl, dataclasses.replace(lay, src_slab=pageable))
    with pytest.raises(R.ReshardError) as e:
        R.reshard_execute(plan, sp, dp)
    assert e.value.code == R.RESHARD_ERR_INVALID_ARG and "pageable" in str(e.value)
    # the plan stays usable with valid pointers afterwards
    sp, dp = R.workload_pointers(wl, lay)
    R.reshard_execute(plan, sp, dp, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert_matches_oracle(wl, lay)


def test_misaligned_items_take_the_staged_kernel_or_the_general_walker():
    """Misaligned items of many short rows in device memory run in the bulk-staged kernel when
    some group has two or more replicas or the rows move at least 512 MB; short single-replica
    launches, and the same items over page-locked host memory (no bulk copies there), in
    reshard_copy_rows_kernel; misaligned single long rows in reshard_copy_kernel; more replicas
    than a staged descriptor holds in the general walker too. All bit-exact."""
    import dataclasses
    # whole source rows (a (2, 1) mesh) into a 3-way column split: destination pitch 2732 bytes
    wl = S.mesh2d_to_1d(rows=512, cols=4096, variant="2d", src_cols=1)      # 2 replicas
    lay, plan = run_gpu(wl)
    st = R.reshard_plan_stats(plan)
    assert st["last_staged_items"] > 0 and st["last_general_items"] == 0
    assert_matches_oracle(wl, lay)
    hl = dataclasses.replace(lay, dst_slab=torch.empty(lay.dst_slab.numel(), dtype=torch.uint8, pin_memory=True))
    hl.dst_slab.fill_(0xA5)
    sp, dp = R.workload_pointers(wl, hl)
    R.reshard_execute(plan, sp, dp, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    st = R.reshard_plan_stats(plan)
    assert st["last_staged_items"] == 0 and st["last_general_items"] > 0 and st["last_rows_kernel"] == 1
    assert_matches_oracle(wl, hl)
    wl = S.mesh2d_to_1d(rows=512, cols=4096, variant="1d", src_cols=1)      # one replica, 8 MB: many-rows walker
    lay, plan = run_gpu(wl)
    st = R.reshard_plan_stats(plan)
    assert st["last_staged_items"] == 0 and st["last_general_items"] > 0 and st["last_rows_kernel"] == 1
    assert_matches_oracle(wl, lay)
    wl = S.dense_ffn(layers=1, hidden=256, ffn=1000)               # contiguous runs, shifted by 2
    lay, plan = run_gpu(wl, misalign=2)
    st = R.reshard_plan_stats(plan)
    assert st["last_general_items"] > 0 and st["last_rows_kernel"] == 0
    assert_matches_oracle(wl, lay)
    wl = _one((96, 333), (2,), ("S0",), (2, 12), ("S1", "R"))     # 12 replicas of 167/166-column rows
    lay, plan = run_gpu(wl)
    st = R.reshard_plan_stats(plan)
    assert st["last_staged_items"] == 0 and st["last_general_items"] > 0
    assert_matches_oracle(wl, lay)


def test_staged_kernel_row_shapes():
    """The staged kernel over rows of every phase pair: source and destination offsets and
    pitches that are not multiples of 16 bytes, runs from 1 to 4096 bytes, 2 to 8 replicas (odd
    counts drain a pair of equal-phase replicas together and the last one alone), many rows per
    stage and one row per stage."""
    cases = [
        _one((300, 2048), (1,), ("R",), (3, 3), ("S1", "R")),         # 683/682-column rows, 3 replicas
        _one((64, 4096), (1,), ("R",), (3, 2), ("S1", "R")),          # rows close to the 4 KiB limit
        _one((500, 9), (1,), ("R",), (2, 2), ("S1", "R")),            # 4-5 element rows, 2 replicas
        _one((200, 1000), (3,), ("S0",), (2, 3), ("R", "S1"), dtype="u8"),
        _one((77, 702), (2,), ("S1",), (5, 3), ("S1", "R"), dtype="f32"),   # 564-byte rows
        _one((40, 130), (1,), ("R",), (8, 2), ("R", "S1")),           # 8 replicas: the staged maximum
    ]
    for wl in cases:
        for mis in (0, 2, 6):
            if mis % S.DTYPES[wl.tensors[0].dtype][1]:
                continue
            lay, plan = run_gpu(wl, misalign=mis)
            assert R.reshard_plan_stats(plan)["last_staged_items"] > 0 or mis == 0
            assert_matches_oracle(wl, lay)


def test_staged_kernel_single_replica_at_size():
    """One replica: the staged kernel takes the rows once they move 512 MB or more (here the
    (2,1) -> (3,) mesh reshard at 4x the rows, 940 MB read + written); compared whole."""
    wl = S.mesh2d_to_1d(rows=57344, variant="1d", src_cols=1)
    lay, plan = run_gpu(wl)
    assert R.reshard_plan_stats(plan)["last_staged_items"] > 0
    assert_matches_oracle(wl, lay)


def _split(shape, ns, nd, reps=1, dtype="bf16", shift=0, dim=-1):
    """`ns` source shards along `dim` into `nd` destination shards along it, each destination
    replicated `reps` times; replica j of a destination starts `shift * j` elements into its
    buffer (replicas whose rows differ in phase mod 16 bytes)."""
    d = len(shape) + dim if dim < 0 else dim
    dm, dp = ((nd, reps), (f"S{d}", "R")) if reps > 1 else ((nd,), (f"S{d}",))
    t = S.TensorDesc("w", shape, dtype, (ns,), (f"S{d}",), dm, dp, [S.View(i) for i in range(ns)],
                     [S.View(i, shift * (i % reps)) for i in range(nd * reps)], seed=43)
    return S.workloads._size_buffers(S.Workload("split", [t]), ns, nd * reps)


def _split_padded_outer(shape, ns, nd):
    """`_split` along the last dim of a 3-D tensor with every destination's outer stride padded
    by 8 elements (its outer dim cannot merge into the rows)."""
    wl = _split(shape, ns, nd)
    t = wl.tensors[0]
    cols = [len(range(*sl)) for sl in _chunks(shape[-1], nd)]
    t.dst_views = [S.View(i, 0, (shape[1] * c + 8, c, 1)) for i, c in enumerate(cols)]
    return S.workloads._size_buffers(S.Workload("split_padded", [t]), ns, nd)


def _chunks(n, k):
    c = -(-n // k)
    return [(min(i * c, n), min((i + 1) * c, n)) for i in range(k)]


GATHER_CASES = {
    "mesh_pieces_2048_684": lambda: _split((300, 4096), 4, 3),
    "two_replicas": lambda: _split((257, 1000), 4, 3, reps=2),
    "replicas_out_of_phase": lambda: _split((129, 1000), 4, 3, reps=2, shift=3),
    "three_replicas_out_of_phase": lambda: _split((65, 1000), 4, 3, reps=3, shift=5),
    "pieces_of_two_elements": lambda: _split((64, 18), 9, 2),             # 4-byte pieces, 18-byte rows
    "u8_odd": lambda: _split((77, 333), 4, 3, reps=2, dtype="u8"),
    "f32": lambda: _split((90, 702), 2, 5, dtype="f32"),                # pairs only across the middle
    "i64_rows": lambda: _split((40, 301), 4, 3, dtype="i64"),
    "three_dims": lambda: _split((3, 50, 1000), 4, 3),
    "four_dims_merged": lambda: _split((2, 3, 20, 1000), 4, 3),
    "outer_stride_padded": lambda: _split_padded_outer((16, 3, 1000), 4, 3),
    "long_rows": lambda: _split((16, 40000), 4, 3, reps=2),              # 26.7 KB rows
    "rows_of_four_pieces": lambda: _split((64, 888), 8, 2),              # two pairs per row
    "rows_of_three_pieces": lambda: _split((64, 999), 9, 3, reps=2),     # a pair and a plain piece
}


@pytest.mark.parametrize("misalign", [0, 2, 6])
@pytest.mark.parametrize("name", sorted(GATHER_CASES))
def test_gather_rows_bit_exact(name, misalign):
    """Destination rows assembled from two source pieces run in reshard_copy_gather_kernel: every
    piece length (4 bytes up), element sizes 1 to 8, replicas in and out of phase, outer dims,
    rows longer than a warp's pass; buffers shifted by 0, 2 or 6 bytes. Bit-exact, canary intact."""
    wl = GATHER_CASES[name]()
    if misalign % S.DTYPES[wl.tensors[0].dtype][1]:
        pytest.skip("shift not a multiple of the element size")
    lay, plan = run_gpu(wl, misalign=misalign)
    n_direct, n_pack, n_unpack = (len(R.reshard_plan_items(plan, k)[0]) for k in (6, 7, 8))
    st = R.reshard_plan_stats(plan)
    assert n_direct > 0 and st["last_gather_items"] == n_direct and st["gather_items"] == n_direct + n_pack + n_unpack
    assert_matches_oracle(wl, lay)
    # packed: the pack pass (scatter items where one source row feeds two message blocks), then
    # the unpack pass's gather items out of the messages
    lay, plan = run_gpu(wl, mode="packed", misalign=misalign, plan=plan)
    assert n_unpack > 0 and R.reshard_plan_stats(plan)["last_gather_items"] == n_pack + n_unpack
    assert_matches_oracle(wl, lay)


def test_gather_items_follow_pointer_changes():
    """The resolved gather table is rebuilt whenever the pointers change: one plan executed on
    three layouts (shifted by 0, 6 and 0 bytes, the last with new buffers), each checked whole,
    and a repeat with unchanged pointers."""
    wl = S.mesh2d_to_1d(rows=143, cols=409, variant="2d")
    lay1, plan = run_gpu(wl)
    assert_matches_oracle(wl, lay1)
    lay2, _ = run_gpu(wl, plan=plan, misalign=6)
    assert_matches_oracle(wl, lay2)
    lay3, _ = run_gpu(wl, plan=plan)
    assert_matches_oracle(wl, lay3)
    S.fill_canary(lay3)
    sp, dp = R.workload_pointers(wl, lay3)
    R.reshard_execute(plan, sp, dp, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert R.reshard_plan_stats(plan)["last_gather_items"] > 0
    assert_matches_oracle(wl, lay3)


def test_gather_items_carry_the_whole_mesh_reshard():
    """The (2,4) -> (3,) and (3,2) mesh reshards: every destination row is two source pieces, so
    the gather kernel is the pass's only launch; the allocation-free entry point walks the same
    plan's plain items and gives the same bytes."""
    for variant in ("1d", "2d"):
        wl = S.mesh2d_to_1d(rows=1434, cols=4096, variant=variant)
        lay, plan = run_gpu(wl)
        st = R.reshard_plan_stats(plan)
        assert st["last_launches"] == 1 and st["last_gather_items"] == len(R.reshard_plan_items(plan, 6)[0]) > 0
        assert st["last_aligned_items"] + st["last_staged_items"] + st["last_general_items"] == 0
        assert_matches_oracle(wl, lay)


def test_readme_example():
    """The usage example of the README, verbatim in substance: 2 row shards -> 4 column shards."""
    from torch.distributed.tensor import Shard
    spec = R.Spec((8, 8), "bf16", (2,), [Shard(0)], (4,), [Shard(1)])
    src = [torch.randn(4, 8, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    dst = [torch.empty(8, 2, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    plan = R.reshard_plan_create(spec)
    R.reshard_execute(plan, src, dst, mode="direct", quant="none",
                      stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(dst, 1), torch.cat(src, 0))


def test_plan_released_right_after_execute():
    """A plan handle dropped while its execute is still queued (garbage-collected at once):
    destroy waits for the device, so the result is complete and correct."""
    import gc
    wl = S.dense_ffn(layers=1, hidden=256, ffn=1000)
    lay = S.allocate(wl, "cuda")
    S.fill_sources(wl, lay)
    S.fill_canary(lay)
    sp, dp = R.workload_pointers(wl, lay)
    R.reshard_execute(R.plan_workload(wl), sp, dp, stream=torch.cuda.current_stream().cuda_stream)
    gc.collect()
    torch.cuda.synchronize()
    assert_matches_oracle(wl, lay)


def test_transposing_items_of_two_element_sizes_take_two_launches():
    wl = SMALL["transpose_mixed_bf16_f32_one_plan"]()
    lay, plan = run_gpu(wl)
    st = R.reshard_plan_stats(plan)
    assert st["last_launches"] == 2 and st["last_aligned_items"] + st["last_general_items"] == 0
    assert_matches_oracle(wl, lay)
