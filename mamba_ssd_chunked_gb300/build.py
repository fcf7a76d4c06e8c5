"""Build libssd.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

    python -m mamba_ssd_chunked_gb300.build [--verbose] [--debug]

Each .cu file under csrc/ compiles in parallel to an object in _build/, then
nvcc links them (static cudart) into mamba_ssd_chunked_gb300/libssd.so.
--debug builds libssd_debug.so instead (objects in _build_debug/), with
SSD_DEBUG defined: every index the tensor-core kernels compute by hand is
checked before use (SSD_CHECK in csrc/ptx.cuh; ssd_debug_build in ssd.h).
"""
from __future__ import annotations

import argparse
import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBRARY = os.path.join(PKG, "libssd.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIBRARY_DEBUG = os.path.join(PKG, "libssd_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _compile(src: str, verbose: bool, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
           "-I", INCLUDE, "-I", CSRC, *extra, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def up_to_date(library: str = LIBRARY) -> bool:
    if not os.path.exists(library):
        return False
    t = os.path.getmtime(library)
    return all(os.path.getmtime(f) <= t for f in sources() + headers() + [__file__])


def build(force: bool = False, verbose: bool = False, extra=(), debug: bool = False) -> str:
    library = LIBRARY_DEBUG if debug else LIBRARY
    build_dir = BUILD_DEBUG if debug else BUILD
    extra = tuple(extra) + (("-DSSD_DEBUG",) if debug else ())
    if not force and up_to_date(library):
        return library
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, extra, build_dir), srcs))
    tmp = library + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, library)
    return library


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true", help="build libssd_debug.so (SSD_DEBUG index checks)")
    a = ap.parse_args()
    print(build(force=a.force or a.verbose, verbose=a.verbose, debug=a.debug))
