"""Compile the CUDA libraries of the package in-tree for sm_103a.

``libkda_spec.so``   the verify walk, rollback and accept (C ABI of include/kda_spec.h)
``libkda_synth.so``  the device side of the seeded input generator (synth.py)

Translation units compile in parallel with nvcc, then link; the outputs land in
``speculative_decode_verify_kda_gb300/_lib`` (git-ignored).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]

LIBS = {
    "libkda_spec.so": ["kda_scan.cu", "spec_accept.cu", "spec_sampled.cu", "kda_round.cpp", "kda_abi.cpp"],
    "libkda_synth.so": ["synth_fill.cu"],
}


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def _compile(src: str, verbose_ptxas: bool) -> tuple[str, str]:
    obj = os.path.join(OBJ_DIR, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVFLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas and src.endswith(".cu"):
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose_ptxas: bool = False) -> dict:
    """Build both libraries; returns {library: path}.  ptxas reports go to stdout if asked."""
    os.makedirs(LIB_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    srcs = sorted({s for v in LIBS.values() for s in v})
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = dict(zip(srcs, ex.map(lambda s: _compile(s, verbose_ptxas), srcs)))
    if verbose_ptxas:
        for s in srcs:
            if results[s][1]:
                print(f"== {s}\n{results[s][1]}")
    out = {}
    for lib, parts in LIBS.items():
        path = os.path.join(LIB_DIR, lib)
        tmp = f"{path}.{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[results[p][0] for p in parts]]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {lib} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
        out[lib] = path
    return out


if __name__ == "__main__":
    import sys
    print(build(verbose_ptxas="-v" in sys.argv))
