"""Compile the in-tree CUDA library (libtcgemm.so) for sm_103a with nvcc.

The translation units compile in parallel, one -gencode, no cmake: the
same commands run on the x86 development machine (cross-compilation, no GPU
needed) and on the Arm GPU machines.  The result lands in ``_build/`` next to this file.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
SO_PATH = os.path.join(OUT_DIR, "libtcgemm.so")
# The debug build: the same sources with the kernel's device-side checks
# (TCG_DEBUG_CHECKS), selected by TCG_DEBUG=1 in the environment.
DEBUG_SO_PATH = os.path.join(OUT_DIR, "libtcgemm_debug.so")


def debug_requested() -> bool:
    return os.environ.get("TCG_DEBUG", "") == "1"


def so_path(debug: bool | None = None) -> str:
    return DEBUG_SO_PATH if (debug_requested() if debug is None else debug) else SO_PATH
GENCODE = "arch=compute_103a,code=sm_103a"
UNITS = ("tcgemm_host", "launch_block_scaled", "launch_grouped", "launch_narrow", "launch_swapped", "debug_tma")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtcgemm.so")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  [os.path.join(ROOT, "include", "tcgemm.h")])


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Build libtcgemm.so, or with debug (default: TCG_DEBUG=1 in the
    environment) libtcgemm_debug.so, unless it is newer than every source."""
    debug = debug_requested() if debug is None else debug
    target = so_path(debug)
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = sources()
    if not force and os.path.exists(target):
        newest = max(os.path.getmtime(s) for s in srcs)
        if os.path.getmtime(target) >= newest:
            return target
    tmp = target + f".tmp{os.getpid()}"
    flags = ["-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
             "-Xptxas", "-v" if verbose else "-O3"] + (["-DTCG_DEBUG_CHECKS"] if debug else [])
    # The kernel's instantiations are split over these translation units,
    # compiled in parallel, then linked into one shared library.
    objs, procs = [], []
    for unit in UNITS:
        obj = os.path.join(OUT_DIR, f"{unit}{'.debug' if debug else ''}.{os.getpid()}.o")
        objs.append(obj)
        procs.append(subprocess.Popen([_nvcc(), *flags, "-c", "-o", obj, os.path.join(CSRC, f"{unit}.cu")]))
    failed = [UNITS[i] for i, pr in enumerate(procs) if pr.wait() != 0]
    try:
        if failed:
            raise RuntimeError(f"nvcc failed on {', '.join(failed)}")
        subprocess.run([_nvcc(), "-gencode", GENCODE, "-shared", "-o", tmp, *objs], check=True)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    os.replace(tmp, target)
    return target
