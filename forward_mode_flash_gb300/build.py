"""Builds the in-tree CUDA library ``_build/libjvp_attn.so`` for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then
linked into one shared library exporting the C ABI of ``include/jvp_attn.h``.
The CUDA runtime is linked statically, so the library loads without a GPU.
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libjvp_attn.so")
# Debug build: device-side bounds checks (-DJVP_DEBUG_CHECKS), built on request only.
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libjvp_attn_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return exe


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + [os.path.join(ROOT, "include", "jvp_attn.h"),
                                      os.path.join(CSRC, "exports.map")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra=(), debug: bool = False) -> str:
    """Compile every translation unit and link the library; returns its path.

    debug=True builds the separate debug library (DEBUG_LIB) whose
    tensor-core kernels bounds-check their hand-computed indices."""
    lib, out_dir = (DEBUG_LIB, DEBUG_BUILD) if debug else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    objs = []
    cmds = []
    defs = ["-DJVP_DEBUG_CHECKS"] if debug else []
    for src in _sources():
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *FLAGS, *defs, *extra, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    workers = min(len(cmds), os.cpu_count() or 4)
    failed = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for cmd, r in ex.map(run, cmds):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = lib + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map"),
            "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
