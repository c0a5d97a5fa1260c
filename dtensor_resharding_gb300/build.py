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


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libreshard.so."""
    srcs = _sources()
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(s) for s in srcs)):
        return LIB_PATH
    bdir = os.path.join(HERE, "_build")
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    jobs = [
        [nvcc, *common, "-x", "c++", "-c", os.path.join(CSRC, "plan.cpp"), "-o", os.path.join(bdir, "plan.o")],
        [nvcc, *common, *ARCH, "-lineinfo", "-Xptxas", "-v" if verbose else "-O3",
         "-c", os.path.join(CSRC, "execute.cu"), "-o", os.path.join(bdir, "execute.o")],
    ]
    procs = [subprocess.Popen(j, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True) for j in jobs]
    logs = []
    for j, p in zip(jobs, procs):
        out, _ = p.communicate()
        logs.append(out)
        if p.returncode:
            raise RuntimeError(f"build failed: {' '.join(j)}\n{out}")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, "-shared", *ARCH, os.path.join(bdir, "plan.o"), os.path.join(bdir, "execute.o"), "-o", tmp]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print("".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
