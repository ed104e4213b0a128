"""Builds libmoe.so in-tree with nvcc for sm_103a (no cmake, no torch
extension machinery): one nvcc per translation unit, run in parallel, then a
shared-library link against the shared CUDA runtime."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe.so")
# Checked build: every row index read from a routing table is verified against
# its buffer before use (MOE_ECORRUPT); a separate library and object folder.
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmoe_checked.so")
SOURCES = ["route_count.cu", "route_split.cu", "route_cluster.cu", "route_pack.cu", "route_pack_fp8.cu", "dispatch_pack.cu", "dispatch_fp8.cu", "dispatch_staged.cu", "dense_a2a.cu", "combine.cu", "combine_two_level.cu", "moe_abi.cu", "moe_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe.so")


def _cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra_flags: Optional[List[str]] = None,
          checked: bool = False) -> str:
    """Compile csrc/*.cu into libmoe.so next to this file (libmoe_checked.so
    with checked=True); returns its path."""
    lib = LIB_CHECKED if checked else LIB
    build_dir = BUILD_CHECKED if checked else BUILD
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input() and not extra_flags:
        return lib
    nv = nvcc()
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
                    "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC] + list(extra_flags or [])
    if checked:
        flags.append("-DMOE_CHECKED")

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nv] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    libdir = _cuda_lib_dir(nv)
    cmd = [nv] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", f"-rpath,{libdir}", "-L", libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
