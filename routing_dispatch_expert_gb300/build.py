"""Build libmoe_gb300.so in-tree with nvcc for sm_103a (one -gencode, sources compiled in parallel)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
SO = os.path.join(OUT_DIR, "libmoe_gb300.so")
SOURCES = ["api.cu", "route.cu", "dispatch.cu", "gemm.cu", "gemm_pair.cu", "gemm_fp8.cu", "gemm_fp4.cu", "combine.cu", "eplb.cu", "fused.cu"]
HEADERS = ["common.cuh", "gemm_common.cuh", "kernels.h", "device_state.h", "route_impl.cuh", "dispatch_impl.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def _newer(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    include = os.path.join(os.path.dirname(PKG), "include", "moe.h")
    common = [os.path.join(CSRC, h) for h in HEADERS] + [include]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _newer(o, [s] + common):
            jobs.append(["nvcc", *FLAGS, *ARCH, "-c", s, "-o", o])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or r.returncode != 0:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    if force or _newer(SO, objs):
        subprocess.check_call(["nvcc", *ARCH, "-shared", "-cudart", "shared", "-o", SO, *objs])
    return SO


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True))
