"""Seeded synthetic inputs for the optimizer-step tests and benchmark.

The common source of inputs for both sides of every parity test: the host
version (``zgen.c``) feeds the CPU oracle, the CUDA twin (``zgen_cuda.cu``)
fills device buffers with the same bits.  The generator definition is in
``zgen.h``.  This package holds none of the optimizer step's arithmetic.
"""
from __future__ import annotations

import ctypes
import math
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_C_SRC = os.path.join(_HERE, "zgen.c")
_CU_SRC = os.path.join(_HERE, "zgen_cuda.cu")
_HDR = os.path.join(_HERE, "zgen.h")
_HOST_LIB = os.path.join(_HERE, "libzgen.so")
_CUDA_LIB = os.path.join(_HERE, "libzgen_cuda.so")

STREAM_GRAD, STREAM_MASTER, STREAM_SHARD = 1, 2, 3
FP16, BF16 = 0, 1
MASK = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
IRWIN_HALL4_STD = math.sqrt(4 * (65536 ** 2 - 1) / 12)

_lock = threading.Lock()
_host = None
_cuda = None


def _stale(lib, *srcs):
    return not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs)


def build_host(force=False):
    if force or _stale(_HOST_LIB, _C_SRC, _HDR):
        tmp = _HOST_LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                        "-o", tmp, _C_SRC], check=True)
        os.replace(tmp, _HOST_LIB)
    return _HOST_LIB


def cuda_build_cmd(out):
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
            "-Xcompiler", "-fPIC", "-shared", "-o", out, _CU_SRC]


def build_cuda(force=False):
    if shutil.which("nvcc") is None:
        raise RuntimeError("nvcc not found: cannot build the CUDA input generator")
    if force or _stale(_CUDA_LIB, _CU_SRC, _HDR):
        tmp = _CUDA_LIB + f".tmp{os.getpid()}"
        subprocess.run(cuda_build_cmd(tmp), check=True)
        os.replace(tmp, _CUDA_LIB)
    return _CUDA_LIB


def build(force=False):
    build_host(force)
    if shutil.which("nvcc"):
        build_cuda(force)


_P, _I64, _U64, _U32, _F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                            ctypes.c_float)


def host():
    global _host
    with _lock:
        if _host is None:
            L = ctypes.CDLL(build_host())
            L.zgen_key.restype = _U64
            L.zgen_key.argtypes = [_U64, _U32, _U32, _U32]
            L.zgen_f32.argtypes = [_U64, _U32, _U32, _U32, _I64, _I64, _F, _F, _P]
            L.zgen_16.argtypes = [_U64, _U32, _U32, _U32, _I64, _I64, _F, _F, ctypes.c_int, _P]
            L.zgen_ranks_16.argtypes = [_U64, _U32, _U32, ctypes.c_int, _I64, _I64, _I64, _F, _F,
                                        ctypes.c_int, _P]
            L.zgen_16_at.argtypes = [_U64, _U32, _U32, _U32, _P, _I64, _F, _F, ctypes.c_int, _P]
            L.zgen_f32_at.argtypes = [_U64, _U32, _U32, _U32, _P, _I64, _F, _F, _P]
            for f in ("zgen_f32", "zgen_16", "zgen_ranks_16", "zgen_16_at", "zgen_f32_at"):
                getattr(L, f).restype = None
            _host = L
    return _host


def cuda():
    global _cuda
    with _lock:
        if _cuda is None:
            L = ctypes.CDLL(build_cuda())
            L.zgen_cuda_ranks_16.argtypes = [_U64, _U32, _U32, ctypes.c_int, _I64, _I64, _I64, _F,
                                             _F, ctypes.c_int, _P, _P]
            L.zgen_cuda_f32.argtypes = [_U64, _U32, _U32, _U32, _I64, _I64, _F, _F, _P, _P]
            L.zgen_cuda_16.argtypes = [_U64, _U32, _U32, _U32, _I64, _I64, _F, _F, ctypes.c_int,
                                       _P, _P]
            for f in ("zgen_cuda_ranks_16", "zgen_cuda_f32", "zgen_cuda_16"):
                getattr(L, f).restype = ctypes.c_int
            _cuda = L
    return _cuda


def kappa(sigma: float) -> float:
    """Scale that gives the Irwin-Hall(4) integer a standard deviation sigma
    (computed in double, rounded once to binary32)."""
    return float(np.float32(sigma / IRWIN_HALL4_STD))


def _ptr(a):
    assert a.flags.c_contiguous
    return a.ctypes.data


# ---- host ---------------------------------------------------------------
def ranks_16(seed, stream, step, nd, n, sigma, scale=1.0, dtype=FP16, rank_stride=None,
             index0=0):
    rs = n if rank_stride is None else rank_stride
    out = np.empty((nd, rs), np.uint16)
    host().zgen_ranks_16(seed, stream, step, nd, index0, n, rs, kappa(sigma), scale, dtype,
                         _ptr(out))
    return out


def ranks_16_mt(seed, stream, step, nd, n, sigma, scale=1.0, dtype=FP16, rank_stride=None,
                index0=0, nthreads=None):
    """ranks_16 with one host thread per rank row (same bits)."""
    import concurrent.futures
    rs = n if rank_stride is None else rank_stride
    out = np.zeros((nd, rs), np.uint16)
    L, k = host(), kappa(sigma)

    def row(r):
        L.zgen_16(seed, stream, step, r, index0, n, k, scale, dtype, out[r].ctypes.data)
    with concurrent.futures.ThreadPoolExecutor(nthreads or min(nd, os.cpu_count() or 1)) as ex:
        list(ex.map(row, range(nd)))
    return out


def f32(seed, stream, step, rank, n, sigma, scale=1.0, index0=0):
    out = np.empty(n, np.float32)
    host().zgen_f32(seed, stream, step, rank, index0, n, kappa(sigma), scale, _ptr(out))
    return out


def s16(seed, stream, step, rank, n, sigma, scale=1.0, dtype=FP16, index0=0):
    out = np.empty(n, np.uint16)
    host().zgen_16(seed, stream, step, rank, index0, n, kappa(sigma), scale, dtype, _ptr(out))
    return out


def s16_at(seed, stream, step, rank, idx, sigma, scale=1.0, dtype=FP16):
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.uint16)
    host().zgen_16_at(seed, stream, step, rank, _ptr(idx), idx.size, kappa(sigma), scale, dtype,
                      _ptr(out))
    return out


def f32_at(seed, stream, step, rank, idx, sigma, scale=1.0):
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.float32)
    host().zgen_f32_at(seed, stream, step, rank, _ptr(idx), idx.size, kappa(sigma), scale,
                       _ptr(out))
    return out


# ---- device (raw pointers; cuda_stream is a cudaStream_t as an int) -------
def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: CUDA error {rc}")


def cuda_ranks_16(out_ptr, seed, stream, step, nd, n, sigma, scale=1.0, dtype=FP16,
                  rank_stride=None, index0=0, cuda_stream=0):
    rs = n if rank_stride is None else rank_stride
    _check(cuda().zgen_cuda_ranks_16(seed, stream, step, nd, index0, n, rs, kappa(sigma), scale,
                                     dtype, out_ptr, cuda_stream), "zgen_cuda_ranks_16")


def cuda_f32(out_ptr, seed, stream, step, rank, n, sigma, scale=1.0, index0=0, cuda_stream=0):
    _check(cuda().zgen_cuda_f32(seed, stream, step, rank, index0, n, kappa(sigma), scale, out_ptr,
                                cuda_stream), "zgen_cuda_f32")


def cuda_s16(out_ptr, seed, stream, step, rank, n, sigma, scale=1.0, dtype=FP16, index0=0,
             cuda_stream=0):
    _check(cuda().zgen_cuda_16(seed, stream, step, rank, index0, n, kappa(sigma), scale, dtype,
                               out_ptr, cuda_stream), "zgen_cuda_16")


# ---- pure-Python statement of the key (for the tests) -----------------
def mix(z: int) -> int:
    z &= MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def key(seed, stream, step, rank) -> int:
    k = mix(seed ^ ((stream * GOLDEN) & MASK))
    k = mix(k + step * GOLDEN)
    return mix(k + rank * GOLDEN)


def inf_site(seed: int, step: int, psi: int, nd: int):
    """Where the overflow test plants +inf at a given step: (rank, index)."""
    index = mix(key(seed, 4, step, 0) + GOLDEN) % psi
    rank = mix(key(seed, 4, step, 1) + GOLDEN) % nd
    return int(rank), int(index)
