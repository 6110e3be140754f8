"""Build libw4a16.so in-tree for sm_103a with nvcc (no cmake).

Each .cu under csrc/ compiles to an object in parallel, then nvcc links the
shared library next to this file. Objects go to <repo>/_build/.

`build(debug=True)` makes the bounds-checking build, libw4a16_debug.so
(compiled with W4A16_DEBUG: kernels check their computed indices and record
W4A16_ERR_BOUNDS instead of making an out-of-bounds access); the binding
loads it when W4A16_LIBRARY names it.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libw4a16.so")
LIB_DEBUG = os.path.join(HERE, "libw4a16_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, extra, bdir: str) -> str:
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip() and os.environ.get("W4A16_BUILD_VERBOSE"):
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, extra=(), debug: bool = False) -> str:
    bdir = os.path.join(BUILD, "debug") if debug else BUILD
    out = LIB_DEBUG if debug else LIB
    os.makedirs(bdir, exist_ok=True)
    extra = list(extra) + (["-DW4A16_DEBUG"] if debug else [])
    if verbose:
        extra += ["-Xptxas", "-v"]
        os.environ["W4A16_BUILD_VERBOSE"] = "1"
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, bdir), srcs))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-lpthread", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug="--debug" in sys.argv))
