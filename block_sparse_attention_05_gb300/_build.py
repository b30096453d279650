"""Builds the in-tree C-ABI library ``_lib/libmsa.so`` for sm_103a with nvcc.

Each translation unit under ``csrc/`` is compiled in parallel to an object file,
then linked into one shared library (static CUDA runtime).  Objects are rebuilt
only when a source or header is newer.
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
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libmsa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=None) -> str:
    os.makedirs(os.path.join(LIB_DIR, "obj"), exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = _headers()
    exe = nvcc()
    # MSA_EXTRA_NVCC_FLAGS adds flags to every compile (e.g. "-DMSA_CHECKED=1" for the checked build)
    flags = FLAGS + os.environ.get("MSA_EXTRA_NVCC_FLAGS", "").split() + list(extra_flags or [])
    # objects built with other flags are stale
    stamp = os.path.join(LIB_DIR, "obj", "flags.txt")
    key = " ".join(ARCH + flags)
    if not os.path.exists(stamp) or open(stamp).read() != key:
        for o in glob.glob(os.path.join(LIB_DIR, "obj", "*.o")):
            os.remove(o)
        if os.path.exists(LIB):
            os.remove(LIB)
        with open(stamp, "w") as f:
            f.write(key)

    def compile_one(src):
        obj = os.path.join(LIB_DIR, "obj", os.path.basename(src) + ".o")
        if _stale(obj, [src] + hdrs):
            cmd = [exe] + ARCH + flags + ["-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if _stale(LIB, objs):
        cmd = [exe] + ARCH + ["-shared", "-o", LIB] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
