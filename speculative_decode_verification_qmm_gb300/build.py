"""Build ``libqmm.so`` in-tree for sm_103a.

Each CUDA translation unit compiles in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``), then nvcc links the
shared library into ``speculative_decode_verification_qmm_gb300/_build/``.
A rebuild happens only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libqmm.so")

SOURCES = ["qmm_api.cu", "qmm_aux.cu", "qmm_verify_q4.cu", "qmm_verify_fp8.cu", "qmm_verify_q8.cu",
           "qmm_verify_tc.cu", "qmm_prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES]
            + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + [os.path.join(INCLUDE, "qmm.h")])


def up_to_date(lib: str | None = None) -> bool:
    lib = LIB if lib is None else lib
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir=None) -> str:
    """Compile the CUDA library if needed and return the path of ``libqmm.so``.

    ``out_dir``: build a variant (for example with ``extra_flags=["-DQMM_TRACE"]``)
    into that folder instead (one set of flags per folder: the up-to-date check
    compares times only); the in-tree library is untouched."""
    lib = LIB if out_dir is None else os.path.join(out_dir, "libqmm.so")
    odir = OUT_DIR if out_dir is None else out_dir
    if not force and up_to_date(lib):
        return lib
    os.makedirs(odir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for s in SOURCES:
        obj = os.path.join(odir, s.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, s), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                          text=True)))
    errors = []
    for s, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {s} ---\n{out}")
        elif verbose and out.strip():
            print(out, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else []))
