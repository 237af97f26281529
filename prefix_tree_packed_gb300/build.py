"""Build the C-ABI library ``libtreeattn.so`` in-tree for sm_103a (GB300).

Every translation unit under ``csrc/`` is compiled in parallel (nvcc for
``.cu``, g++ for host-only ``.cpp``) and linked into one shared library next
to this file.  CUDA runtime is linked statically, so loading the library on a
machine without a GPU works (the planner runs on the host alone).

Usage:  python prefix_tree_packed_gb300/build.py [-v]   (run as a file: importing the
package itself needs the built library)
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libtreeattn.so")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.isdir(c):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("CUDA toolkit not found (set CUDA_HOME)")


def _sources():
    srcs = sorted(os.listdir(CSRC))
    return [os.path.join(CSRC, s) for s in srcs if s.endswith((".cu", ".cpp"))]


def _compile(src: str, cuda: str, verbose: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda, "include")]
    if src.endswith(".cu"):
        cmd = [os.path.join(cuda, "bin", "nvcc"), "-O3", "-std=c++17", *ARCH, "-lineinfo",
               "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xptxas", "-v" if verbose else "-O3", *inc, "-c", src, "-o", obj]
    else:
        cmd = ["g++", "-O3", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-Wall", *inc, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, file=sys.stderr)
    return obj


def build(verbose: bool = False) -> str:
    cuda = _cuda_home()
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, cuda, verbose), srcs))
    tmp = OUT + ".tmp"
    cmd = [os.path.join(cuda, "bin", "nvcc"), "-shared", *ARCH, "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
