"""Build libqsa.so (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m sparse_attention_long_qsa_gb300.build [--force] [--verbose]

Translation units compile in parallel into _build/ at the repository root and
link into sparse_attention_long_qsa_gb300/libqsa.so.  The runtime is linked
shared (libcudart.so.13), so a process that already loaded PyTorch's CUDA
runtime shares it.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "qsa")
LIB = os.path.join(PKG, "libqsa.so")
SOURCES = ["api.cu", "pool.cu", "index.cu", "attn.cu", "attn_pf.cu", "attn_union.cu", "append.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return hdrs + [os.path.abspath(__file__)]


def _stale(target: str, inputs) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    deps = _deps()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        if force or _stale(o, [s] + deps):
            jobs.append([nvcc] + flags + ["-c", s, "-o", o])

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, p in ex.map(run, jobs):
                if verbose or ptxas_verbose or p.returncode:
                    sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
                if p.returncode:
                    raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    objs = [os.path.join(BUILD, s + ".o") for s in SOURCES]
    if force or jobs or _stale(LIB, objs):
        libdir = _cuda_lib_dir(nvcc)
        tmp = LIB + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", f"-rpath,{libdir}", "-Xlinker", "-rpath,$ORIGIN"]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or p.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + p.stdout + p.stderr)
        if p.returncode:
            raise RuntimeError("link of libqsa.so failed")
        os.replace(tmp, LIB)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose))


if __name__ == "__main__":
    main()
