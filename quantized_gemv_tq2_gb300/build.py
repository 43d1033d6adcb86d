"""Build the CUDA library in-tree: quantized_gemv_tq2_gb300/_lib/libtq2_gb300.so,
and its bounds-checked debug variant _lib/check/libtq2_gb300.so.

Each translation unit is compiled in parallel for sm_103a only, then linked
into one shared library exporting the C ABI of include/tq2.h.  The CUDA
runtime is linked statically, so the library needs only the driver at run
time.  The debug variant is compiled with TQ2_BOUNDS_CHECK: the kernels check
their computed global and shared-memory indices, skip an access that would
fall outside its buffer and report it as TQ2_FLAG_BOUNDS in the caller's
status word (nothing traps).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtq2_gb300.so")
OBJ_DIR = os.path.join(LIB_DIR, "obj")
CHECK_DIR = os.path.join(LIB_DIR, "check")
CHECK_LIB_PATH = os.path.join(CHECK_DIR, "libtq2_gb300.so")

NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-Xptxas", "-v",
    "-I", os.path.join(ROOT, "include"),
]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "tq2.h"), os.path.abspath(__file__)]


def lib_path(bounds_check: bool = False) -> str:
    return CHECK_LIB_PATH if bounds_check else LIB_PATH


def up_to_date(bounds_check: bool = False) -> bool:
    path = lib_path(bounds_check)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _start(bounds_check: bool, nvcc: str):
    obj_dir = os.path.join(CHECK_DIR, "obj") if bounds_check else OBJ_DIR
    os.makedirs(obj_dir, exist_ok=True)
    extra = ["-DTQ2_BOUNDS_CHECK"] if bounds_check else []
    procs, objs = [], []
    for src in _sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), src, obj + ".log"))
    return procs, objs


def _finish(bounds_check: bool, nvcc: str, procs, objs, verbose: bool) -> str:
    failed = []
    for p, src, log in procs:
        out, _ = p.communicate()
        with open(log, "wb") as f:
            f.write(out)
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose:
            sys.stdout.write(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    path = lib_path(bounds_check)
    tmp = path + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                    *objs, "-o", tmp], check=True)
    os.replace(tmp, path)
    return path


def build(force: bool = False, verbose: bool = False, bounds_check: bool = False, both: bool = False) -> str:
    """Build the release library (or, with bounds_check, the checked one;
    with both, the two at once, every translation unit in parallel).
    Returns the path of the release library (the checked one if only it
    was asked for)."""
    nvcc = os.environ.get("NVCC", "nvcc")
    variants = [False, True] if both else [bounds_check]
    started = []
    for v in variants:
        if force or not up_to_date(v):
            started.append((v, *_start(v, nvcc)))
    for v, procs, objs in started:
        _finish(v, nvcc, procs, objs, verbose)
    return lib_path(bounds_check and not both)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, both="--both" in sys.argv,
                bounds_check="--check" in sys.argv))
