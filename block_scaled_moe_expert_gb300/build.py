"""Compile the CUDA library (csrc/*.cu) for sm_103a into libbsmoe.so, in tree.

Each translation unit is compiled in parallel with nvcc; the objects are
linked into one shared library next to this file. Rebuilds only what changed
(object newer than its source and every header).
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libbsmoe.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def _nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def _headers():
    return glob.glob(os.path.join(SRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(obj, src, newest_header):
    return not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header)


def build(verbose=False, ptxas_verbose=False):
    """Build libbsmoe.so; returns its path. Raises RuntimeError on failure."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(SRC, "*.cu")))
    newest_header = max([os.path.getmtime(h) for h in _headers()] + [0])
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    jobs = []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if ptxas_verbose or _stale(obj, src, newest_header):
            jobs.append([nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj])
    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
            for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
                logs.append(res.stdout + res.stderr)
                if res.returncode != 0:
                    raise RuntimeError("nvcc failed: %s\n%s" % (" ".join(cmd), res.stdout + res.stderr))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources]
    if jobs or not os.path.exists(LIB):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed: %s\n%s" % (" ".join(cmd), res.stdout + res.stderr))
    if verbose:
        for l in logs:
            if l.strip():
                print(l)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
