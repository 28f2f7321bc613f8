"""Build the CUDA library in-tree: ``offload_streamed_gb300/_lib/libtiled_linear.so``.

The translation units (GEMM kernels, the engine's ring, stats, hooks and C
ABI, the allocation-free forward, the host optimizer and the file tier) are compiled in parallel by nvcc for sm_103a only, then linked against the shared CUDA
runtime (the same ``libcudart.so.13`` PyTorch loads, so streams created by
either side are one runtime's streams).  The build is skipped when the shared
library is newer than every source and header.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libtiled_linear.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# host code: no fused multiply-add contraction, so that the host-side
# optimizer update gives the same bits on every host architecture
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-Xcompiler", "-ffp-contract=off", "-I", INCLUDE, "-I", CSRC]
# Extra flags of single units: the host optimizer's row loop vectorizes its
# square roots only without errno semantics.
UNIT_FLAGS = {"tl_adam.cpp": ["-Xcompiler", "-fno-math-errno"]}
UNITS = ["tl_gemm.cu", "tl_static.cu", "tl_ring.cpp", "tl_stats.cpp", "tl_hooks.cpp", "tl_abi.cpp", "tl_adam.cpp",
         "tl_filetier.cpp", "tl_optimizer.cpp"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtiled_linear")


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    os.makedirs(LIBDIR, exist_ok=True)
    cc = nvcc()
    objs, procs = [], []
    for u in UNITS:
        obj = os.path.join(LIBDIR, f"{os.path.splitext(u)[0]}.{os.getpid()}.o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *UNIT_FLAGS.get(u, []), "-c", os.path.join(CSRC, u), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((u, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    errors = []
    for u, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {u} ---\n{out.decode(errors='replace')}")
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB + f".tmp{os.getpid()}"
    libdir = os.path.join(cuda_home(), "lib64")
    link = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    for o in objs:
        if os.path.exists(o):
            os.remove(o)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
