"""bench.py's reference arm on the host: one JSON line with the contract's keys (no GPU)."""
import json
import os
import subprocess
import sys

from conftest import ROOT


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "example_8x8", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    for k in ("metric", "value", "n_gpus", "steps", "warmup", "ms_per_step", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["steps"] == 3 and d["warmup"] == 3 and d["value"] > 0


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_e2e_prefix_keeps_the_longest_prefix_that_fits():
    """The end-to-end leg's host budget: the whole workload when it fits, else the longest
    prefix of tensors whose page-locked slabs fit (one more tensor would not), else none."""
    sys.path.insert(0, ROOT)
    import bench
    import synthetic as S

    def host_bytes(w):
        lay = S.allocate(w, "meta")
        return lay.src_slab.numel() + lay.dst_slab.numel() + (lay.scale_slab.numel() if lay.scale_slab is not None else 0)

    def prefix(wl, k):
        w = S.Workload(wl.name, wl.tensors[:k], wl.quant, wl.values)
        return S.workloads._size_buffers(w, len(wl.src_buffer_numel), len(wl.dst_buffer_numel))

    assert bench.host_ram_bytes() > 0
    for wl in (S.dense_ffn(layers=4, hidden=256, ffn=1024),
               S.moe_experts(layers=2, experts=16, hidden=128, ffn=64, dst="tp4")):
        total = host_bytes(wl)
        w, k = bench.e2e_prefix(wl, total)
        assert w is wl and k == len(wl.tensors)
        for budget in (total // 2, total // 5):
            w, k = bench.e2e_prefix(wl, budget)
            assert 0 < k < len(wl.tensors)
            assert host_bytes(w) <= budget < host_bytes(prefix(wl, k + 1))
            assert [t.name for t in w.tensors] == [t.name for t in wl.tensors[:k]]
        assert bench.e2e_prefix(wl, 16) == (None, 0)
