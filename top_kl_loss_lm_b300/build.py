"""Build libkdtopk.so in-tree with nvcc for sm_103a (B300).

Usage: ``python -m top_kl_loss_lm_b300.build [--force] [-v] [--checked]`` (or
``__graft_entry__.build()``, which builds both). The shared library lands next
to this file, where ``binding`` loads it from. ``--checked`` builds
libkdtopk_checked.so with -DKD_CHECKED: every bulk-tensor copy checks its
coordinates and the selection kernels their slots, recording KD_ERR_BOUNDS
instead of making an out-of-bounds access (a stand-in for a memory sanitizer;
the tests compare it with the normal build).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libkdtopk.so")
LIB_CHECKED = os.path.join(HERE, "libkdtopk_checked.so")
SOURCES = ["kd_lib.cu"]
DEPENDS = ["kd_lib.cu", "kd_gemm.cuh", "kd_aux.cuh", "kd_ptx.cuh", "kd_sched.h", "kd_logits.cuh", "kd_topk_cache.cuh"]
HEADERS = [os.path.join(os.path.dirname(HERE), "include", h)
           for h in ("kd_topk_kl.h", "kd_topk_kl_testing.h")]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def flags() -> list:
    return ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
            "-Xcompiler", "-fPIC,-O2", "-shared", "-cudart", "static"]


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in DEPENDS] + HEADERS
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build_library(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    if not force and not _stale(lib):
        return lib
    tmp = lib + ".tmp"
    cmd = ([nvcc_path()] + flags() + (["-DKD_CHECKED"] if checked else []) + ["-o", tmp]
           + [os.path.join(CSRC, s) for s in SOURCES])
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv,
                        checked="--checked" in sys.argv))
