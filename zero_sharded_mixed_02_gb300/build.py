"""Compile libzero_b200.so in-tree with nvcc for sm_103a.

The translation units are compiled in parallel into ``_build/`` and linked into
``libzero_b200.so`` next to this file.  Nothing is installed.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzero_b200.so")

SOURCES = ["zero_abi.cu", "zero_step_fp16.cu", "zero_step_bf16.cu", "zero_step_q_fp16.cu",
           "zero_step_q_bf16.cu", "zero_gather.cu",
           "zero_noalloc.cu", "zero_qwz.cu", "zero_ckpt.cu", "zero_offload.cu",
           "zero_cpu_adam.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]
# Host-only sources (the ZeRO-Offload host Adam): every floating-point operation
# rounded on its own (no fused multiply-add), which the element loop needs to
# match the device update bit for bit; errno and trap assumptions relaxed so the
# loop vectorises (neither changes a value).  No -march: the same flags build
# on x86-64 and AArch64.
HOST_FLAGS = ["-std=c++17", "-O3", "-ffp-contract=off", "-fno-math-errno", "-fno-trapping-math",
              "-fPIC", "-pthread", "-Wall", "-I", INCLUDE, "-I", CSRC]


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "zero_b200.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    if shutil.which("nvcc") is None:
        raise RuntimeError("nvcc not found: cannot build libzero_b200")
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        if src.endswith(".cpp"):
            cmd = ["g++", *HOST_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        else:
            cmd = ["nvcc", *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                             text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"{src}:\n{out}")
        elif verbose and out:
            print(out, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", *ARCH, "-shared", "-o", tmp, *objs, "-lpthread"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
