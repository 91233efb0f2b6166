"""Build libgdn.so for sm_103a from csrc/ with nvcc (in-tree, no cmake).

Usage: ``python -m gated_deltanet_linear_rule_gb300.build`` or ``build()``.
The translation units compile in parallel; the result is
``gated_deltanet_linear_rule_gb300/_build/libgdn.so``.  ``build(checked=True)`` compiles the
same sources with GDN_CHECKED into ``_build/checked/libgdn_checked.so``: kernels that test
their computed memory ranges before each access and report a failed test in the device status
word (GDN_DEV_BOUNDS) instead of touching memory -- a debug build standing in for a device
memory checker.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libgdn.so")
LIB_CHECKED = os.path.join(BUILD, "checked", "libgdn_checked.so")
SOURCES = ["gdn_pool.cu", "gdn_decode.cu", "gdn_prefill.cu", "gdn_chunk.cu", "gdn_chunk_small.cu", "gdn_proj.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool, checked: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr"]
    if checked:
        f += ["-DGDN_CHECKED"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None, checked: bool = False) -> str:
    """Compile every CUDA translation unit and link libgdn.so (libgdn_checked.so when checked);
    returns the library path."""
    out_dir = os.path.dirname(LIB_CHECKED) if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "gdn.h"))
    cc = nvcc()
    objs, todo = [], []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [sp] + headers):
            todo.append([cc, *_flags(verbose_ptxas, checked), "-c", sp, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    logs = []
    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or len(todo)) as ex:
            logs = list(ex.map(run, todo))
    if force or todo or _stale(lib, objs):
        logs.append(run([cc, *ARCH, "-shared", "-o", lib, *objs]))
    if verbose_ptxas:
        for log in logs:
            sys.stdout.write(log)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv))
