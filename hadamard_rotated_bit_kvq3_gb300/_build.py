"""Builds libkvq3.so in-tree with nvcc for sm_103a (GB300).

Every translation unit is compiled in parallel, then linked into one shared
library next to this file.  No CMake, no torch extension machinery: the
library is a plain C ABI (include/kvq3.h)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libkvq3.so")
BUILD = os.path.join(ROOT, "_build")
# the checked build: every kernel with its bounds checks (KVQ3_CHECKED) on
LIB_CHECKED = os.path.join(HERE, "libkvq3_checked.so")
BUILD_CHECKED = os.path.join(ROOT, "_build", "checked")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
         "-Xptxas", "-warn-spills", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq3.so")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra=(), checked: bool = False) -> str:
    """Compiles (when stale) and links libkvq3.so -- or, with checked=True,
    libkvq3_checked.so, whose kernels carry the bounds checks that report
    KVQ3_DEV_CHECK -- and returns its path."""
    lib_path, build_dir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    if checked:
        extra = (*extra, "-DKVQ3_CHECKED")
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "kvq3.h"))
    objs, jobs = [], []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if _stale(obj, [src] + headers):
            jobs.append([cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj])

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
        if verbose and (p.stdout or p.stderr):
            print(p.stdout + p.stderr, file=sys.stderr)
        return p

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, jobs))
    if jobs or _stale(lib_path, objs):
        run([cc, *ARCH, "-shared", "-o", lib_path, *objs])
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, checked="--checked" in sys.argv))
