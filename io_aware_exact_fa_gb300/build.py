"""Build libfa_gb300.so in-tree with nvcc for sm_103a (no cmake, no torch).

    python -m io_aware_exact_fa_gb300.build [--verbose] [--ptxas-info] [--debug]

Compiles the translation units under csrc/ in parallel into _build/ and
links them (static CUDA runtime) into io_aware_exact_fa_gb300/libfa_gb300.so.
With --debug (debug=True) the same sources are compiled with FA_DEBUG=1 into
_build_debug/ and libfa_gb300_debug.so: the device-checking build.
Rebuilds only when a source or header is newer than the library.
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfa_gb300.so")
LIB_DEBUG = os.path.join(PKG, "libfa_gb300_debug.so")
SOURCES = ["fa_api.cu", "prefill_sm103.cu", "decode_sm103.cu", "backward_sm103.cu", "decode_grouped_sm103.cu",
           "materialized_sm103.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put it on PATH)")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile and link the library (the checking build with debug=True); returns its path."""
    lib = LIB_DEBUG if debug else LIB
    bdir = BUILD + "_debug" if debug else BUILD
    if not force and not ptxas_info and up_to_date(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"] + (["-DFA_DEBUG=1"] if debug else [])
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, cmd, r

    objs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, obj, cmd, r in ex.map(compile_one, SOURCES):
            if verbose or ptxas_info or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}")
            objs.append(obj)
    tmp = lib + ".tmp"
    # cuBLAS (the materialising baseline's GEMMs) is opened at run time with dlopen, not linked
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("link failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the device-checking build (FA_DEBUG=1)")
    a = ap.parse_args()
    print(build(a.verbose, a.ptxas_info, a.force, a.debug))
