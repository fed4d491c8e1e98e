"""Build libteattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu file compiles in its own nvcc process, in parallel, then one link step
per library produces ``bwd_packed_varlen_gb300/lib/libteattn.so`` and its debug
build ``libteattn_debug.so`` (compiled with ``TEATTN_DEBUG_BOUNDS``: every computed
global offset is checked and a bad one is recorded as ``TE_STATUS_OUT_OF_BOUNDS``
in the call's status word instead of being accessed). Objects go to ``_build/``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "lib", "libteattn.so")
LIB_DEBUG = os.path.join(PKG, "lib", "libteattn_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]
VARIANTS = {"release": (LIB, []), "debug": (LIB_DEBUG, ["-DTEATTN_DEBUG_BOUNDS"])}


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(job) -> str:
    src, variant, verbose = job
    obj = os.path.join(BUILD, variant, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *VARIANTS[variant][1], "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, variants=("release", "debug")) -> str:
    """Compile every kernel source for each variant and link the shared libraries;
    returns the path of the release library."""
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    srcs = _sources()
    jobs = []
    for v in variants:
        os.makedirs(os.path.join(BUILD, v), exist_ok=True)
        jobs += [(s, v, verbose and v == "release") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(_compile, jobs))
    for v in variants:
        lib = VARIANTS[v][0]
        vobjs = [o for o, j in zip(objs, jobs) if j[1] == v]
        tmp = lib + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *vobjs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
