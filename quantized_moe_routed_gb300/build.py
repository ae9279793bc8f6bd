"""Build the sm_103a C-ABI library libmoe_nvfp4.so in-tree (nvcc, no cmake).

The four translation units compile in parallel, then link into
quantized_moe_routed_gb300/_build/libmoe_nvfp4.so (static cudart).  The
compiler's output for each unit (the kernels' ptxas register and spill report)
is kept beside the objects as <unit>.log.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmoe_nvfp4.so")
SOURCES = ("moe_kernels.cu", "moe_tc.cu", "moe_small.cu", "moe_gemv.cu", "moe_route.cu", "moe_abi.cu")
HEADERS = ("moe_internal.h", "moe_device.cuh", "moe_tcgen05.cuh")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "moe_nvfp4.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-diag-suppress", "128",
              "-I", os.path.join(ROOT, "include"), "-I", CSRC] + ARCH
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if src in ("moe_kernels.cu", "moe_tc.cu", "moe_small.cu", "moe_gemv.cu", "moe_route.cu"):
            cmd += ["-Xptxas", "-v"]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        with open(os.path.join(BUILD, src + ".log"), "w") as f:
            f.write(out)
        if verbose or pr.returncode:
            sys.stderr.write(out)
        if pr.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, "-shared", "-o", tmp] + objs + ARCH, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
