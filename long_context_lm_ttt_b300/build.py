"""Build the CUDA library libttt.so in-tree with nvcc for sm_103a.

    python -m long_context_lm_ttt_b300.build                 # incremental
    python -m long_context_lm_ttt_b300.build --clean         # from scratch
    python -m long_context_lm_ttt_b300.build --debug-bounds  # libttt_debug.so

The debug library is the same sources compiled with TTT_DEBUG_BOUNDS: the
range checks of csrc/bounds.cuh record a violation and skip the access
instead of running it.  Setting TTT_LIBRARY=debug makes the binding load it.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libttt.so")
BUILD_DEBUG = os.path.join(ROOT, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libttt_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def _newer(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(clean: bool = False, verbose: bool = False, extra=None, debug_bounds: bool = False) -> str:
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    if clean and os.path.isdir(build_dir):
        shutil.rmtree(build_dir)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    extra = list(extra or []) + (["-DTTT_DEBUG_BOUNDS"] if debug_bounds else [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        if not clean and not _newer(obj, [src] + headers):
            return obj, None
        cmd = [NVCC] + ARCH + FLAGS + extra + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            return obj, r.stderr + r.stdout
        if verbose and (r.stderr or r.stdout):
            print(r.stderr + r.stdout, flush=True)
        return obj, None

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    errs = [e for _, e in results if e]
    if errs:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errs))
    objs = [o for o, _ in results]
    if _newer(lib, objs):
        cmd = [NVCC] + ARCH + ["-shared", "-o", lib] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stderr + r.stdout)
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--clean", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register/smem usage")
    ap.add_argument("--debug-bounds", action="store_true", help="build libttt_debug.so with the range checks")
    a = ap.parse_args()
    extra = ["-Xptxas", "-v"] if a.ptxas_info else []
    print(build(clean=a.clean or a.ptxas_info, verbose=a.verbose or a.ptxas_info, extra=extra,
                debug_bounds=a.debug_bounds))


if __name__ == "__main__":
    sys.exit(main())
