"""Builds libspecverify.so in-tree for sm_103a (nvcc + g++, five translation
units compiled in parallel, no cmake).  Run as ``python -m
speculative_decoding_verification_14_gb300.build`` or through ``build()``."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libspecverify.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ("spec_verify.cu", "greedy.cu", "truncated.cu")
HOST_SOURCES = ("planner.cpp", "adapt.cpp")
SOURCES = [os.path.join(CSRC, f) for f in (*CUDA_SOURCES, "sv_internal.h", *HOST_SOURCES)] + [
    os.path.join(INCLUDE, "spec_verify.h")]


def _nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def stale() -> bool:
    if not os.path.exists(OUT):
        return True
    t = os.path.getmtime(OUT)
    return any(os.path.getmtime(s) > t for s in SOURCES)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return OUT
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    obj_cu = [os.path.join(BUILD_DIR, f.replace(".cu", ".o")) for f in CUDA_SOURCES]
    obj_cpp = [os.path.join(BUILD_DIR, f.replace(".cpp", ".o")) for f in HOST_SOURCES]
    cmds = [
        [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "-c", os.path.join(CSRC, f), "-o", o] for f, o in zip(CUDA_SOURCES, obj_cu)
    ] + [["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-c",
          os.path.join(CSRC, f), "-o", o] for f, o in zip(HOST_SOURCES, obj_cpp)]
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT) for c in cmds]
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError("build failed: " + " ".join(c) + "\n" + out.decode(errors="replace"))
        if verbose and out:
            sys.stdout.write(out.decode(errors="replace"))
    tmp = OUT + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *obj_cu, *obj_cpp]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed: " + " ".join(link) + "\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
