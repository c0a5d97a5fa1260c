"""Build libreshard.so in-tree: host planner (C++) + device executor (CUDA, sm_103a only)."""
from __future__ import annotations

import os
import shutil
import subprocess
from typing import List

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB_PATH = os.path.join(HERE, "libreshard.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    return shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"


def _sources() -> List[str]:
    out = []
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cpp", ".cu", ".h", ".cuh")):
                out.append(os.path.join(d, f))
    return out


def build(force: bool = False, verbose: bool = False, extra_flags: List[str] = (), out: str = LIB_PATH) -> str:
    """Compile (if stale) and return the path of libreshard.so.

    ``extra_flags`` (or RESHARD_EXTRA_NVCC_FLAGS, space separated) are appended to the CUDA
    compile, e.g. -DRESHARD_UNROLL=8 for launch-shape sweeps; they force a rebuild."""
    extra = list(extra_flags) + os.environ.get("RESHARD_EXTRA_NVCC_FLAGS", "").split()
    force = force or bool(extra)
    srcs = _sources()
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(s) for s in srcs)):
        return out
    tag = "" if out == LIB_PATH else os.path.basename(out).replace(".so", "")
    bdir = os.path.join(HERE, "_build", tag)
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    jobs = [
        [nvcc, *common, *extra, "-x", "c++", "-c", os.path.join(CSRC, "plan.cpp"), "-o", os.path.join(bdir, "plan.o")],
        [nvcc, *common, *ARCH, "-lineinfo", "-Xptxas", "-v" if verbose else "-O3", *extra,
         "-c", os.path.join(CSRC, "execute.cu"), "-o", os.path.join(bdir, "execute.o")],
    ]
    procs = [subprocess.Popen(j, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True) for j in jobs]
    logs = []
    for j, p in zip(jobs, procs):
        log, _ = p.communicate()
        logs.append(log)
        if p.returncode:
            raise RuntimeError(f"build failed: {' '.join(j)}\n{log}")
    tmp = out + f".tmp{os.getpid()}"
    link = [nvcc, "-shared", *ARCH, os.path.join(bdir, "plan.o"), os.path.join(bdir, "execute.o"), "-o", tmp]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}")
    os.replace(tmp, out)
    if verbose:
        print("".join(logs))
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
