"""Build the CUDA library in-tree: quantized_gemv_tq2_gb300/_lib/libtq2_gb300.so,
its bounds-checked debug variant _lib/check/libtq2_gb300.so and, on demand,
its trace variant _lib/trace/libtq2_gb300.so.

Each translation unit is compiled in parallel for sm_103a only, then linked
into one shared library exporting the C ABI of include/tq2.h.  The CUDA
runtime is linked statically, so the library needs only the driver at run
time.  The debug variant is compiled with TQ2_BOUNDS_CHECK: the kernels check
their computed global and shared-memory indices, skip an access that would
fall outside its buffer and report it as TQ2_FLAG_BOUNDS in the caller's
status word (nothing traps).  The trace variant is compiled with TQ2_TRACE:
the class-column kernel stamps the GPU timer at its phase points
(tq2_trace_read); it is for measuring where a call's time goes, never for
timing.
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
TRACE_DIR = os.path.join(LIB_DIR, "trace")
TRACE_LIB_PATH = os.path.join(TRACE_DIR, "libtq2_gb300.so")
# variant -> (library, object directory, extra nvcc flags)
VARIANTS = {
    "release": (LIB_PATH, OBJ_DIR, []),
    "check": (CHECK_LIB_PATH, os.path.join(CHECK_DIR, "obj"), ["-DTQ2_BOUNDS_CHECK"]),
    "trace": (TRACE_LIB_PATH, os.path.join(TRACE_DIR, "obj"), ["-DTQ2_TRACE"]),
}

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


def _variant(bounds_check: bool = False, variant: str | None = None) -> str:
    return variant or ("check" if bounds_check else "release")


def lib_path(bounds_check: bool = False, variant: str | None = None) -> str:
    return VARIANTS[_variant(bounds_check, variant)][0]


def up_to_date(bounds_check: bool = False, variant: str | None = None) -> bool:
    path = lib_path(bounds_check, variant)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _start(variant: str, nvcc: str):
    _, obj_dir, extra = VARIANTS[variant]
    os.makedirs(obj_dir, exist_ok=True)
    procs, objs = [], []
    for src in _sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), src, obj + ".log"))
    return procs, objs


def _finish(variant: str, nvcc: str, procs, objs, verbose: bool) -> str:
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
    path = VARIANTS[variant][0]
    tmp = path + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                    *objs, "-o", tmp], check=True)
    os.replace(tmp, path)
    return path


def build(force: bool = False, verbose: bool = False, bounds_check: bool = False, both: bool = False,
          variant: str | None = None) -> str:
    """Build the release library (or the variant asked for: bounds_check or
    variant "check" / "trace"; with both, the release and the checked
    libraries at once, every translation unit in parallel).  Returns the
    path of the library asked for (the release one with both)."""
    nvcc = os.environ.get("NVCC", "nvcc")
    want = _variant(bounds_check, variant)
    variants = ["release", "check"] if both else [want]
    started = []
    for v in variants:
        if force or not up_to_date(variant=v):
            started.append((v, *_start(v, nvcc)))
    for v, procs, objs in started:
        _finish(v, nvcc, procs, objs, verbose)
    return lib_path(variant="release" if both else want)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, both="--both" in sys.argv,
                bounds_check="--check" in sys.argv, variant="trace" if "--trace" in sys.argv else None))
