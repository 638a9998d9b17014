"""Compile libringattn.so and its check build in-tree for sm_103a (nvcc, every
translation unit of both in parallel).

    python -m online_softmax_attention_zigzag_gb300.build [-v]

Objects go to ``_build/release`` and ``_build/check`` at the repository root; the
libraries land next to this file, where the Python binding loads them:
libringattn.so, and libringattn_check.so (-DRA_CHECK: the kernels check the memory
indices they derive and record RA_ERR_BOUNDS instead of going out of bounds; the binding
loads it when RINGATTN_CHECK=1).
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
LIB = os.path.join(PKG, "libringattn.so")
LIB_CHECK = os.path.join(PKG, "libringattn_check.so")  # -DRA_CHECK: index checks in the kernels
SOURCES = ["api.cu", "attn_bf16.cu", "attn_f32.cu", "permute_merge.cu", "ulysses.cu", "attn_bwd.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return r.returncode, r.stdout


def _objects(nvcc, variant, extra):
    """(source, command, object) for every translation unit of one library variant."""
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, variant, src.replace(".cu", ".o"))
        jobs.append((src, [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj], obj))
    return jobs


def build(verbose: bool = False) -> str:
    """Compile libringattn.so and the check build libringattn_check.so (-DRA_CHECK: index
    checks that record RA_ERR_BOUNDS), all translation units of both in parallel."""
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []
    variants = {"release": (LIB, []), "check": (LIB_CHECK, ["-DRA_CHECK"])}
    jobs = {}
    for name, (_, defs) in variants.items():
        os.makedirs(os.path.join(BUILD, name), exist_ok=True)
        jobs[name] = _objects(nvcc, name, [*defs, *extra])
    flat = [j for js in jobs.values() for j in js]
    with ThreadPoolExecutor(max_workers=len(flat)) as ex:
        results = list(ex.map(lambda j: (j[0], *_run(j[1])), flat))
    failed = False
    for src, rc, out in results:
        if rc != 0 or verbose:
            sys.stdout.write(f"== {src} (rc={rc})\n{out}")
        failed |= rc != 0
    if failed:
        raise RuntimeError("nvcc failed")
    for name, (lib, _) in variants.items():
        tmp = lib + ".tmp"
        rc, out = _run([nvcc, *ARCH, "-shared", "-o", tmp, *[j[2] for j in jobs[name]]])
        if rc != 0:
            sys.stdout.write(out)
            raise RuntimeError("link failed")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
