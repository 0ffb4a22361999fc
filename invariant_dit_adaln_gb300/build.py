"""Build libadaln.so in-tree with nvcc for sm_103a (GB300).

The translation units are compiled in parallel and linked into
``invariant_dit_adaln_gb300/lib/libadaln.so`` (git-ignored).  Flags:
``-gencode arch=compute_103a,code=sm_103a -O3 -lineinfo --fmad=false``; no
fast math, so every floating-point operation rounds as written.
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
BUILD = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libadaln.so")
SOURCES = ["api.cu", "out.cu", "proj.cu", "tc_proj.cu", "res.cu", "f32.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "--fmad=false", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xptxas", "-warn-spills", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libadaln.so")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "adaln.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str | None = None) -> str:
    """Compile and link the library; returns its path.  `variant` names a test
    build with extra flags, linked to lib/<variant>/libadaln.so with objects in
    _build/<variant>/ (the release library is lib/libadaln.so)."""
    lib = LIB if variant is None else os.path.join(LIBDIR, variant, "libadaln.so")
    objdir = BUILD if variant is None else os.path.join(BUILD, variant)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    logs = "".join(log for _, log in results)
    if verbose and logs.strip():
        print(logs, file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


# Test build: the first wait of every waiting kernel goes to an mbarrier that
# nothing arrives on, with a 200 us limit (the kernels' time-out path).
WAIT_TEST_FLAGS = ["-DADALN_TEST_WAIT_NEVER_NS=200000"]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
