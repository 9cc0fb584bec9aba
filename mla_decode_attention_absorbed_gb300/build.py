"""Build the in-tree CUDA library ``libmla.so`` for sm_103a with nvcc.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object file,
then one link step makes the shared library next to this file.  The CUDA
runtime is linked statically, so the library loads without a libcudart on the
loader path (the driver itself is only needed once a call runs).
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
LIB = os.path.join(PKG, "libmla.so")
OBJ_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the MLA library cannot be built")
    return p


def _flags(debug: bool = False):
    f = ARCH + ["-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    f += ["-O0", "-G"] if debug else ["-O3"]
    return f


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + [
        os.path.join(ROOT, "include", "mla.h"), os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra: list | None = None) -> str:
    """Compile (if stale) and return the path of libmla.so."""
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    cc = nvcc()
    flags = _flags() + list(extra or [])
    jobs = []
    for src in _sources():
        obj = os.path.join(OBJ_DIR, os.path.basename(src)[:-3] + ".o")
        jobs.append((src, obj, [cc, "-c", src, "-o", obj] + flags))

    def run(job):
        src, obj, cmd = job
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        return src, r.returncode, r.stdout

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(run, jobs))
    failed = [(s, out) for s, rc, out in results if rc != 0]
    if verbose or failed:
        for s, rc, out in results:
            if out.strip():
                print(f"--- {os.path.basename(s)} (rc={rc})\n{out}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(s) for s, _ in failed))
    tmp = LIB + ".tmp"
    link = [cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [o for _, o, _ in jobs] + ["-lcuda"] * 0
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
