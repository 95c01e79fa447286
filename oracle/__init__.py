"""Plain CPU oracle of the ZeRO-DP sharded mixed-precision optimizer step.

TEST INFRASTRUCTURE ONLY.  The C source (``zero_oracle.c``) is the slow,
obviously-correct statement of what the GPU library computes; this module
builds it with gcc and wraps it with ctypes/numpy.  Only the test suite, the
package entry point's smoke check and the benchmark's CPU-baseline leg may
import it.  It shares nothing with the CUDA library and never imports it.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_HDR = os.path.join(_HERE, "zero_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")

# gcc flags: binary32 evaluation, no contraction into fused multiply-add, no
# fast-math, so each float operation in the source is one IEEE rounding.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
          "-fPIC", "-shared", "-pthread"]

FP16, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc); returns its path."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("decoupled_wd", ctypes.c_int), ("clip_norm", ctypes.c_float),
                ("dynamic_scale", ctypes.c_int), ("backoff", ctypes.c_float),
                ("growth_interval", ctypes.c_int), ("skip_on_overflow", ctypes.c_int)]


class Scalars(ctypes.Structure):
    _fields_ = [("loss_scale", ctypes.c_float), ("good_steps", ctypes.c_int32),
                ("t", ctypes.c_int64), ("beta1_pow", ctypes.c_double),
                ("beta2_pow", ctypes.c_double)]


class Result(ctypes.Structure):
    _fields_ = [("skipped", ctypes.c_int32), ("overflow", ctypes.c_int32),
                ("grad_norm", ctypes.c_double), ("clip_coef", ctypes.c_float),
                ("bc1", ctypes.c_float), ("bc2", ctypes.c_float)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


@dataclasses.dataclass
class Opt:
    """Optimizer description in plain Python (mirrors ``zo_hparams``)."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    decoupled_wd: int = 1
    clip_norm: float = 0.0
    dynamic_scale: int = 0
    backoff: float = 0.5
    growth_interval: int = 1000
    skip_on_overflow: int = 0

    def c(self) -> Hparams:
        return Hparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                       self.decoupled_wd, self.clip_norm, self.dynamic_scale,
                       self.backoff, self.growth_interval, self.skip_on_overflow)


def new_scalars(loss_scale: float = 1.0) -> Scalars:
    return Scalars(loss_scale, 0, 0, 1.0, 1.0)


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_D = ctypes.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # ZO_ORACLE_LIB lets the mutation test load a copy with a planted mistake
            L = ctypes.CDLL(os.environ.get("ZO_ORACLE_LIB") or build())
            sig = {
                "zo_half_to_float": (ctypes.c_float, [ctypes.c_uint16]),
                "zo_float_to_half": (ctypes.c_uint16, [ctypes.c_float]),
                "zo_bf16_to_float": (ctypes.c_float, [ctypes.c_uint16]),
                "zo_float_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "zo_to_float_n": (None, [ctypes.c_int, _P, _P, _I64]),
                "zo_from_float_n": (None, [ctypes.c_int, _P, _P, _I64]),
                "zo_state_bytes": (_D, [_D, _D, ctypes.c_int, _D]),
                "zo_comm_volume": (_D, [_D, _D, ctypes.c_int, ctypes.c_int]),
                "zo_max_params": (_D, [_D, _D, ctypes.c_int, _D]),
                "zo_shard_elems": (_I64, [_I64, ctypes.c_int]),
                "zo_reduce": (ctypes.c_int, [ctypes.c_int, _I64, ctypes.c_int, _P, _I64,
                                             ctypes.c_float, _P]),
                "zo_sumsq": (_D, [_I64, _P]),
                "zo_clip_coef": (ctypes.c_float, [_D, ctypes.c_float]),
                "zo_advance": (None, [_P, _P, ctypes.c_int, _P]),
                "zo_adam": (None, [_I64, _P, ctypes.c_float, _P, _P, _P, _P, ctypes.c_int,
                                   _P, ctypes.c_float, ctypes.c_float]),
                "zo_step": (ctypes.c_int, [ctypes.c_int, _I64, ctypes.c_int, _P, _P, _P, _P,
                                           _P, _P, _P, _P]),
                "zo_step_sharded": (ctypes.c_int, [ctypes.c_int, _I64, _I64, ctypes.c_int, _P,
                                                   _P, _P, _P, _P, _P, _P, _P, ctypes.c_int]),
                "zo_gather_unit": (None, [ctypes.c_int, _I64, _I64, _P, _P]),
                "zo_quantize_f32": (None, [_P, _I64, ctypes.c_int, _I64, _P, _P]),
                "zo_dequantize_f32": (None, [_P, _P, _I64, ctypes.c_int, _I64, _P]),
                "zo_quantize_16": (None, [ctypes.c_int, _P, _I64, ctypes.c_int, _I64, _P, _P]),
                "zo_dequantize_16": (None, [ctypes.c_int, _P, _P, _I64, ctypes.c_int, _I64, _P]),
                "zo_gather_unit_q": (None, [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64,
                                            ctypes.c_int, _I64, _P, _P, _P]),
                "zo_shard_unit": (None, [ctypes.c_int, _I64, _I64, _P, _P]),
                "zo_layout_shard_len": (_I64, [_P]),
                "zo_layout_global": (_I64, [_P, ctypes.c_int, _I64]),
                "zo_reshard": (None, [_P, _P, _P, _P, ctypes.c_int]),
                "zo_reduce16": (ctypes.c_int, [ctypes.c_int, _I64, ctypes.c_int, _P, _I64,
                                               ctypes.c_float, _P, _P]),
                "zo_step_offload": (ctypes.c_int, [ctypes.c_int, _I64, ctypes.c_int, _P, _P, _P,
                                                   _P, _P, _P, _P, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


# ---- 16-bit formats -------------------------------------------------------
def to_float(dtype: int, bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float32)
    lib().zo_to_float_n(dtype, _ptr(bits), _ptr(out), bits.size)
    return out


def from_float(dtype: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().zo_from_float_n(dtype, _ptr(x), _ptr(out), x.size)
    return out


# ---- ledger ---------------------------------------------------------------
def state_bytes(psi, nd, stage, K=12):
    return lib().zo_state_bytes(float(psi), float(nd), stage, float(K))


def comm_volume(psi, nd, stage, exact=0):
    return lib().zo_comm_volume(float(psi), float(nd), stage, int(exact))


def max_params(mem_bytes, nd, stage, K=12):
    return lib().zo_max_params(float(mem_bytes), float(nd), stage, float(K))


def shard_elems(psi, nd):
    return lib().zo_shard_elems(int(psi), int(nd))


# ---- step stages ------------------------------------------------------------
def reduce(nd, dtype, grads, loss_scale=1.0, n=None, rank_stride=None):
    """Stages 1-2 on grads[nd][...]; returns (g float32[n], overflow)."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    rs = grads.shape[-1] if rank_stride is None else rank_stride
    n = rs if n is None else n
    g = np.empty(n, np.float32)
    ovf = lib().zo_reduce(nd, n, dtype, _ptr(grads), rs, loss_scale, _ptr(g))
    return g, bool(ovf)


def sumsq(g):
    g = np.ascontiguousarray(g, dtype=np.float32)
    return lib().zo_sumsq(g.size, _ptr(g))


def clip_coef(norm, clip):
    return lib().zo_clip_coef(norm, clip)


def advance(opt: Opt, st: Scalars, overflow: bool) -> Result:
    hp, res = opt.c(), Result()
    lib().zo_advance(ctypes.addressof(hp), ctypes.addressof(st), int(overflow),
                     ctypes.addressof(res))
    return res


def adam(g, c, master, m, v, params, dtype, opt: Opt, bc1, bc2):
    hp = opt.c()
    lib().zo_adam(g.size, _ptr(g), c, _ptr(master), _ptr(m), _ptr(v), _ptr(params), dtype,
                  ctypes.addressof(hp), bc1, bc2)


def step(nd, dtype, grads, master, m, v, params, opt: Opt, st: Scalars) -> dict:
    """Unsharded definition; updates master/m/v/params/st in place."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    n = master.size
    assert grads.shape == (nd, n) and m.size == n and v.size == n and params.size == n
    hp, res = opt.c(), Result()
    rc = lib().zo_step(nd, n, dtype, _ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                       ctypes.addressof(hp), ctypes.addressof(st), ctypes.addressof(res))
    if rc != 0:
        raise MemoryError("oracle step: allocation failed")
    return res.as_dict()


def reduce16(nd, dtype, grads, loss_scale=1.0, n=None, rank_stride=None):
    """The offloaded reduce: returns (g16 uint16[n] as copied to the host,
    g float32[n] unscaled on the host, overflow)."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    rs = grads.shape[-1] if rank_stride is None else rank_stride
    n = rs if n is None else n
    g16 = np.empty(n, np.uint16)
    g = np.empty(n, np.float32)
    ovf = lib().zo_reduce16(nd, n, dtype, _ptr(grads), rs, loss_scale, _ptr(g16), _ptr(g))
    return g16, g, bool(ovf)


def step_offload(nd, dtype, grads, master, m, v, params, opt: Opt, st: Scalars) -> dict:
    """One ZeRO-Offload step; updates master/m/v/params/st in place."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    n = master.size
    assert grads.shape == (nd, n) and m.size == n and v.size == n and params.size == n
    hp, res = opt.c(), Result()
    rc = lib().zo_step_offload(nd, n, dtype, _ptr(grads), _ptr(master), _ptr(m), _ptr(v),
                               _ptr(params), ctypes.addressof(hp), ctypes.addressof(st),
                               ctypes.addressof(res))
    if rc != 0:
        raise MemoryError("oracle offload step: allocation failed")
    return res.as_dict()


def step_sharded(nd, dtype, grads, master, m, v, params, opt: Opt, st: Scalars,
                 shard=None, nthreads=1) -> dict:
    """Sharded execution of the same step (rank r owns [r*shard, (r+1)*shard))."""
    grads = np.ascontiguousarray(grads, dtype=np.uint16)
    n = master.size
    assert grads.shape == (nd, n)
    shard = shard_elems(n, nd) if shard is None else shard
    hp, res = opt.c(), Result()
    rc = lib().zo_step_sharded(nd, n, shard, dtype, _ptr(grads), _ptr(master), _ptr(m), _ptr(v),
                               _ptr(params), ctypes.addressof(hp), ctypes.addressof(st),
                               ctypes.addressof(res), nthreads)
    if rc != 0:
        raise MemoryError("oracle step: allocation failed")
    return res.as_dict()


# ---- ZeRO-3 unit gather ---------------------------------------------------
def gather_unit(nd, length, slice_elems, slices):
    slices = [np.ascontiguousarray(s, dtype=np.uint16) for s in slices]
    ptrs = (ctypes.c_void_p * nd)(*[_ptr(s) for s in slices])
    out = np.zeros(length, np.uint16)
    lib().zo_gather_unit(nd, length, slice_elems, ctypes.addressof(ptrs), _ptr(out))
    return out


def shard_unit(nd, unit, slice_elems):
    unit = np.ascontiguousarray(unit, dtype=np.uint16)
    slices = [np.empty(slice_elems, np.uint16) for _ in range(nd)]
    ptrs = (ctypes.c_void_p * nd)(*[_ptr(s) for s in slices])
    lib().zo_shard_unit(nd, unit.size, slice_elems, _ptr(unit), ctypes.addressof(ptrs))
    return slices


# ---- sharded checkpoint: regrouping shards for another layout ---------------
class _Layout(ctypes.Structure):
    _fields_ = [("nd", ctypes.c_int), ("nunits", ctypes.c_int), ("len", ctypes.c_void_p)]


class Layout:
    """nd ranks over units of the given lengths (stages 0-2: one unit of psi)."""

    def __init__(self, nd, unit_lens):
        self.nd = int(nd)
        self.lens = np.ascontiguousarray(np.asarray(unit_lens, dtype=np.int64))
        self.c = _Layout(self.nd, int(self.lens.size), _ptr(self.lens))

    @property
    def psi(self):
        return int(self.lens.sum())

    def shard_len(self):
        return int(lib().zo_layout_shard_len(ctypes.byref(self.c)))

    def global_index(self, r, j):
        return int(lib().zo_layout_global(ctypes.byref(self.c), r, j))


def reshard(A, old_shards, B):
    """old_shards: A.nd arrays of A.shard_len() elements (one dtype) -> B.nd arrays."""
    old = [np.ascontiguousarray(x) for x in old_shards]
    dt = old[0].dtype
    assert all(x.dtype == dt and x.size == A.shard_len() for x in old) and len(old) == A.nd
    new = [np.empty(B.shard_len(), dt) for _ in range(B.nd)]
    for x in new:                                   # nonzero fill: padding must be written
        x.view(np.uint8)[:] = 0xA5
    po = (ctypes.c_void_p * A.nd)(*[_ptr(x) for x in old])
    pn = (ctypes.c_void_p * B.nd)(*[_ptr(x) for x in new])
    lib().zo_reshard(ctypes.byref(A.c), ctypes.addressof(po), ctypes.byref(B.c),
                     ctypes.addressof(pn), dt.itemsize)
    return new


# ---- ZeRO++ qwZ block quantization ----------------------------------------
def code_bytes(n, bits):
    return n if bits == 8 else (n + 1) // 2


def quantize_f32(x, bits=8, block=256):
    x = np.ascontiguousarray(x, np.float32)
    q = np.zeros(code_bytes(x.size, bits), np.uint8)
    scales = np.zeros(-(-x.size // block), np.float32)
    lib().zo_quantize_f32(_ptr(x), x.size, bits, block, _ptr(q), _ptr(scales))
    return q, scales


def dequantize_f32(q, scales, n, bits=8, block=256):
    out = np.empty(n, np.float32)
    lib().zo_dequantize_f32(_ptr(np.ascontiguousarray(q)), _ptr(np.ascontiguousarray(scales)), n,
                            bits, block, _ptr(out))
    return out


def quantize_16(dtype, x, bits=8, block=256):
    x = np.ascontiguousarray(x, np.uint16)
    q = np.zeros(code_bytes(x.size, bits), np.uint8)
    scales = np.zeros(-(-x.size // block), np.float32)
    lib().zo_quantize_16(dtype, _ptr(x), x.size, bits, block, _ptr(q), _ptr(scales))
    return q, scales


def dequantize_16(dtype, q, scales, n, bits=8, block=256):
    out = np.empty(n, np.uint16)
    lib().zo_dequantize_16(dtype, _ptr(np.ascontiguousarray(q)), _ptr(np.ascontiguousarray(scales)),
                           n, bits, block, _ptr(out))
    return out


def gather_unit_q(dtype, nd, length, slice_elems, offset, bits, block, qs, scales):
    qs = [np.ascontiguousarray(q, np.uint8) for q in qs]
    scales = [np.ascontiguousarray(s, np.float32) for s in scales]
    qp = (ctypes.c_void_p * nd)(*[_ptr(q) for q in qs])
    sp = (ctypes.c_void_p * nd)(*[_ptr(s) for s in scales])
    out = np.zeros(length, np.uint16)
    lib().zo_gather_unit_q(dtype, nd, length, slice_elems, offset, bits, block,
                           ctypes.addressof(qp), ctypes.addressof(sp), _ptr(out))
    return out
