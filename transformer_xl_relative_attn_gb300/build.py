"""Builds libtxl.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each .cu under csrc/ compiles to an object in _build/ in parallel; the objects
link into transformer_xl_relative_attn_gb300/libtxl.so.  The bounds-checked
variant (every computed kernel index checked, -DTXL_CHECKED) builds the same
sources into _build/checked/ and libtxl_checked.so.  Rebuilds only what
changed (object older than its source or any header).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtxl.so")
LIB_CHECKED = os.path.join(PKG, "libtxl_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtxl.so")
    return cand


def _deps_mtime() -> float:
    hdrs = (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(INCLUDE, "*.h")))
    return max((os.path.getmtime(h) for h in hdrs), default=0.0)


def _compile(src: str, obj: str, extra: list[str]) -> None:
    cmd = [nvcc(), *ARCH, *NVFLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")


def _jobs(build_dir: str, extra: list[str], force: bool):
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    dep_t = _deps_mtime()
    jobs, objs = [], []
    for s in srcs:
        o = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), dep_t):
            jobs.append((s, o, extra))
    return jobs, objs


def _link(lib: str, objs: list[str], relink: bool) -> None:
    newest = max((os.path.getmtime(o) for o in objs), default=0.0)
    if relink or not os.path.exists(lib) or os.path.getmtime(lib) < newest:
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = True) -> str:
    """Builds libtxl.so and (checked=True) libtxl_checked.so, all objects in
    one parallel pool; returns the path of libtxl.so."""
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    jobs, objs = _jobs(BUILD, extra, force)
    cjobs, cobjs = _jobs(os.path.join(BUILD, "checked"), extra + ["-DTXL_CHECKED"], force) if checked else ([], [])
    todo = jobs + cjobs
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(todo), os.cpu_count() or 4))) as ex:
        for f in [ex.submit(_compile, s, o, e) for s, o, e in todo]:
            f.result()
    _link(LIB, objs, force or bool(jobs))
    if checked:
        _link(LIB_CHECKED, cobjs, force or bool(cjobs))
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas=True))
