"""Builds libpkv.so in-tree from csrc/ with nvcc for sm_103a (no cmake, no torch extension).

Translation units compile in parallel; the library lands in
``paged_kv_cache_73_gb300/lib/libpkv.so``.  A rebuild happens only when a
source or header is newer than the library (or ``force=True``).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libpkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-Wextra"]


def _nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpkv.so")
    return exe


def _cuda_include() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(_nvcc()))), "include")


def sources():
    names = sorted(os.listdir(CSRC))
    return [os.path.join(CSRC, n) for n in names if n.endswith((".cu", ".cpp"))]


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, n) for n in os.listdir(CSRC)] + [os.path.join(INCLUDE, n) for n in os.listdir(INCLUDE)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link libpkv.so; returns its path."""
    if not force and not _stale():
        return LIB_PATH
    nvcc = _nvcc()
    obj_dir = os.path.join(LIB_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    jobs = []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        if src.endswith(".cu"):
            cmd = [nvcc] + CU_FLAGS + ["-I", INCLUDE, "-c", src, "-o", obj]
        else:
            cxx = shutil.which("g++") or "g++"
            cmd = [cxx] + CXX_FLAGS + ["-I", INCLUDE, "-I", _cuda_include(), "-c", src, "-o", obj]
        jobs.append((src, obj, cmd))

    def run(job):
        src, obj, cmd = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(run, jobs))
    failed = [(s, r) for s, r in results if r.returncode != 0]
    for s, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(f"--- {os.path.basename(s)}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("libpkv build failed: " + ", ".join(os.path.basename(s) for s, _ in failed))
    tmp = LIB_PATH + ".tmp"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for _, o, _ in jobs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("libpkv link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
