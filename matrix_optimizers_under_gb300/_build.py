"""In-tree build of libmfsdp.so for sm_103a (nvcc + g++, no cmake).

Each translation unit compiles in parallel; the CUDA runtime is linked
statically so the library loads on a machine without a GPU (the planner and the
argument checks are pure host code and are tested there).
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libmfsdp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC] + ARCH
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    cu = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    cpp = sorted(f for f in os.listdir(CSRC) if f.endswith(".cpp"))
    return cu, cpp


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def needs_build() -> bool:
    """True when the library is missing or older than any source or header."""
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    srcs = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(f) > t for f in srcs)


def ensure_built() -> str:
    return build() if needs_build() else LIB


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every CUDA/C++ source of the library and link libmfsdp.so."""
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = _nvcc()
    cu, cpp = _sources()
    jobs = []
    for f in cu:
        extra = ["-Xptxas", "-v"] if ptxas_verbose else []
        jobs.append([nvcc] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, f), "-o",
                                                   os.path.join(BUILD, f + ".o")])
    for f in cpp:
        jobs.append([os.environ.get("CXX", "g++")] + CXX_FLAGS + ["-c", os.path.join(CSRC, f), "-o",
                                                                  os.path.join(BUILD, f + ".o")])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        outs = list(ex.map(_run, jobs))
    objs = [os.path.join(BUILD, f + ".o") for f in cu + cpp]
    tmp = LIB + ".tmp"
    out = _run([nvcc, "-shared", "-cudart", "static"] + ARCH + ["-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"])
    os.replace(tmp, LIB)
    if verbose:
        for o in outs + [out]:
            if o.strip():
                print(o, file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB)
