"""Build libddt.so in-tree with nvcc for sm_103a (no CMake).

Each .cu under csrc/ is compiled to an object in parallel, then linked into
``tree_speculative_decoding_gb300/libddt.so``.  Objects are rebuilt when a
source or header is newer.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libddt.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                 "--expt-relaxed-constexpr", f"-I{os.path.join(ROOT, 'include')}"]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    jobs = []
    objs = []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if ptxas_info or _stale(obj, [src] + headers):
            cmd = [NVCC] + CFLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", src, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode != 0:
                print(" ".join(cmd))
                print(r.stdout, r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    # objects of sources that no longer exist are dropped, and a changed set of
    # objects relinks even when every remaining object is up to date
    for old in glob.glob(os.path.join(BUILD, "*.o")):
        if old not in objs:
            os.remove(old)
    manifest = os.path.join(BUILD, "objects.txt")
    listed = open(manifest).read().split("\n") if os.path.exists(manifest) else None
    if jobs or _stale(LIB, objs) or listed != objs:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            print(r.stdout, r.stderr)
            raise RuntimeError("link of libddt.so failed")
        os.replace(tmp, LIB)
        with open(manifest, "w") as f:
            f.write("\n".join(objs))
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
