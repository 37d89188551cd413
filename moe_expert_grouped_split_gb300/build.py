"""Build libdwdp.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object in
_build/, then linked into moe_expert_grouped_split_gb300/libdwdp.so (CUDA
runtime linked statically; the driver is reached through
cudaGetDriverEntryPointByVersion, so the library loads on a machine without a
GPU).  Run ``python -m moe_expert_grouped_split_gb300.build`` or call
``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libdwdp.so"
SOURCES = ["gemm.cu", "route.cu", "dwdp_abi.cu", "route_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def _inputs_mtime() -> float:
    files = [CSRC / s for s in SOURCES] + list(CSRC.glob("*.h")) + [PKG.parent / "include" / "dwdp.h",
                                                                     Path(__file__)]
    return max(f.stat().st_mtime for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> Path:
    if not force and LIB.exists() and LIB.stat().st_mtime >= _inputs_mtime():
        return LIB
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str):
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-I", str(PKG.parent / "include"), "-c", str(CSRC / src),
               "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    for src, obj, r in results:
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}")
    tmp = BUILD / "libdwdp.so.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", str(tmp)] + [str(o) for _, o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
