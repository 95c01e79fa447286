"""Python binding of libzero_b200 (declared in include/zero_b200.h).

The ZeRO-DP sharded mixed-precision optimizer step on one GPU: Nd data-parallel
ranks emulated in the GPU's own memory; reduce-scatter, unscale with overflow
skip, global-norm clip, Adam/AdamW, 16-bit cast and the all-gather write-back
(ZeRO-1/2) or the per-unit gather (ZeRO-3), all in the library's CUDA kernels.

Argument marshalling only: every function has the name of the C entry point it
calls.  Device buffers are passed as raw device pointers (ints), or as any
object with a ``data_ptr()`` method (e.g. a torch tensor); streams as
``cudaStream_t`` values (ints).  Non-OK status codes raise ``ZeroError``.
There is no fallback: if the compiled library is missing, loading fails.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence, Tuple

_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_DIR, "libzero_b200.so")

(ZERO_OK, ZERO_EINVAL, ZERO_ENOMEM, ZERO_ECUDA, ZERO_ETIMEOUT, ZERO_ENOENT, ZERO_ECORRUPT,
 ZERO_EIO, ZERO_ESTATE) = range(9)
ZERO_CKPT_FSYNC, ZERO_CKPT_DROP_CACHE = 1, 2
ZERO_FP16, ZERO_BF16 = 0, 1
PATH_FUSED, PATH_G32, PATH_RECOMPUTE = 0, 1, 2

# every entry point declared in include/zero_b200.h
ENTRY_POINTS = (
    "zero_plan_create", "zero_plan_create_units", "zero_plan_destroy", "zero_plan_layout",
    "zero_plan_unit", "zero_step", "zero_step_qwz", "zero_step_pingpong", "zero_plan_state_set",
    "zero_step_result", "zero_step_overflow",
    "zero_gather_layer", "zero_state_bytes", "zero_comm_volume", "zero_max_params",
    "zero_status_string", "zero_plan_profile", "zero_plan_kernel_times", "zero_plan_path",
    "zero_grad_norm_noalloc", "zero_plan_set_reduce_kernel", "zero_quantize_shard",
    "zero_gather_layer_q", "zero_plan_set_bucket", "zero_step_bucket", "zero_step_apply",
    "zero_checkpoint_save", "zero_checkpoint_load", "zero_offload_step", "zero_cpu_adam",
)


class ZeroError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {zero_status_string(code)}")


class zero_hparams_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("decoupled_wd", ctypes.c_int), ("clip_norm", ctypes.c_float),
                ("loss_scale", ctypes.c_float), ("dynamic_scale", ctypes.c_int),
                ("backoff", ctypes.c_float), ("growth_interval", ctypes.c_int),
                ("skip_on_overflow", ctypes.c_int)]


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, decoupled_wd=1,
            clip_norm=0.0, loss_scale=1.0, dynamic_scale=0, backoff=0.5,
            growth_interval=1000, skip_on_overflow=0) -> zero_hparams_t:
    return zero_hparams_t(lr, beta1, beta2, eps, weight_decay, decoupled_wd, clip_norm,
                          loss_scale, dynamic_scale, backoff, growth_interval,
                          skip_on_overflow)


_lock = threading.Lock()
_lib = None
_P, _U64, _I64 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int64
_PU64, _PI64 = ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_int64)


def lib():
    """Load libzero_b200.so (built in-tree by __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libzero_b200 is not built ({LIB_PATH} missing); "
                                  "run __graft_entry__.build() first")
            L = ctypes.CDLL(LIB_PATH)
            st = ctypes.c_int
            sig = {
                "zero_plan_create": (st, [_U64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P,
                                          ctypes.c_int, _P, _P]),
                "zero_plan_create_units": (st, [_U64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                _P, _P, ctypes.c_int, _P, _P, _P]),
                "zero_plan_destroy": (st, [_P]),
                "zero_plan_layout": (st, [_P, _PU64, _PU64, ctypes.POINTER(ctypes.c_int), _PU64]),
                "zero_plan_unit": (st, [_P, ctypes.c_int, _PU64, _PU64, _PU64]),
                "zero_step": (st, [_P, _P, _P, _P, _P, _P, _P, _P]),
                "zero_step_qwz": (st, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P]),
                "zero_step_pingpong": (st, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
                "zero_plan_state_set": (st, [_P, ctypes.POINTER(ctypes.c_int)]),
                "zero_step_result": (st, [_P, ctypes.POINTER(ctypes.c_int),
                                          ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_float),
                                          ctypes.POINTER(ctypes.c_float), _PI64]),
                "zero_step_overflow": (st, [_P, ctypes.POINTER(ctypes.c_int)]),
                "zero_gather_layer": (st, [_P, ctypes.c_int, _P, _P, _P]),
                "zero_state_bytes": (_U64, [_U64, _U64, ctypes.c_int, ctypes.c_int]),
                "zero_comm_volume": (_U64, [_U64, _U64, ctypes.c_int, ctypes.c_int]),
                "zero_max_params": (_U64, [_U64, _U64, ctypes.c_int, ctypes.c_int]),
                "zero_status_string": (ctypes.c_char_p, [ctypes.c_int]),
                "zero_plan_profile": (st, [_P, ctypes.c_int]),
                "zero_plan_kernel_times": (st, [_P, ctypes.POINTER(ctypes.c_double),
                                                ctypes.POINTER(ctypes.c_double), _PI64, _PI64]),
                "zero_plan_path": (ctypes.c_int, [_P]),
                "zero_grad_norm_noalloc": (st, [_P, ctypes.c_int, _U64, _U64, ctypes.c_int,
                                                ctypes.c_float, _P, _P, _P]),
                "zero_plan_set_reduce_kernel": (st, [_P, ctypes.c_int]),
                "zero_quantize_shard": (st, [ctypes.c_int, _P, _U64, ctypes.c_int, _P, _P, _P]),
                "zero_gather_layer_q": (st, [_P, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P]),
                "zero_plan_set_bucket": (st, [_P, _U64, _PU64]),
                "zero_step_bucket": (st, [_P, _U64, _P, _P, _P]),
                "zero_step_apply": (st, [_P, _P, _P, _P, _P, _P, _P]),
                "zero_checkpoint_save": (st, [_P, ctypes.c_char_p, ctypes.c_int, _P, _P, _P, _P,
                                              ctypes.c_int, _P]),
                "zero_checkpoint_load": (st, [_P, ctypes.c_char_p, ctypes.c_int, _P, _P, _P, _P,
                                              _P]),
                "zero_offload_step": (st, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P]),
                "zero_cpu_adam": (st, [_P, ctypes.c_int, _U64, ctypes.c_float, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_float, _P, _P, _P, _P, _P,
                                       ctypes.c_int]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype, fn.argtypes = res, args
            _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _hptr(x) -> Optional[int]:
    """Address of a host array: a numpy array or a CPU tensor."""
    if x is None:
        return None
    if hasattr(x, "__array_interface__"):
        return x.__array_interface__["data"][0]
    return _ptr(x)


def _check(code: int, where: str):
    if code != ZERO_OK:
        raise ZeroError(code, where)


def zero_status_string(code: int) -> str:
    return lib().zero_status_string(code).decode()


def _shape_arrays(shapes: Sequence[Sequence[int]]):
    dims = [int(d) for s in shapes for d in s]
    ndims = [len(s) for s in shapes]
    return ((ctypes.c_int64 * max(1, len(dims)))(*dims),
            (ctypes.c_int * max(1, len(ndims)))(*ndims))


def zero_plan_create(psi: int, nd: int, stage: int, dtype: int, shapes: Sequence[Sequence[int]],
                     hp: zero_hparams_t, units: Optional[Sequence[int]] = None) -> int:
    """Returns an opaque plan handle; ``units`` (stage 3) selects
    zero_plan_create_units."""
    dims, ndims = _shape_arrays(shapes)
    out = ctypes.c_void_p()
    if units is None:
        code = lib().zero_plan_create(psi, nd, stage, dtype, ctypes.addressof(dims),
                                      ctypes.addressof(ndims), len(shapes), ctypes.byref(hp),
                                      ctypes.byref(out))
    else:
        u = (ctypes.c_int * max(1, len(units)))(*units)
        code = lib().zero_plan_create_units(psi, nd, stage, dtype, ctypes.addressof(dims),
                                            ctypes.addressof(ndims), len(shapes),
                                            ctypes.addressof(u), ctypes.byref(hp),
                                            ctypes.byref(out))
    _check(code, "zero_plan_create")
    return out.value


def zero_plan_create_units(psi, nd, stage, dtype, shapes, units, hp) -> int:
    return zero_plan_create(psi, nd, stage, dtype, shapes, hp, units=units)


def zero_plan_destroy(plan: int) -> None:
    _check(lib().zero_plan_destroy(plan), "zero_plan_destroy")


def zero_plan_layout(plan: int) -> Tuple[int, int, int, int]:
    """(shard_elems, padded_elems, nunits, workspace_bytes)"""
    s, p, w = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    u = ctypes.c_int()
    _check(lib().zero_plan_layout(plan, ctypes.byref(s), ctypes.byref(p), ctypes.byref(u),
                                  ctypes.byref(w)), "zero_plan_layout")
    return s.value, p.value, u.value, w.value


def zero_plan_unit(plan: int, unit: int) -> Tuple[int, int, int]:
    """(len, slice_elems, offset) of a ZeRO-3 unit"""
    n, s, o = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib().zero_plan_unit(plan, unit, ctypes.byref(n), ctypes.byref(s), ctypes.byref(o)),
           "zero_plan_unit")
    return n.value, s.value, o.value


def zero_plan_path(plan: int) -> int:
    return lib().zero_plan_path(plan)


REDUCE_LDG, REDUCE_TMA = 0, 1


def zero_plan_set_reduce_kernel(plan: int, kind: int) -> None:
    _check(lib().zero_plan_set_reduce_kernel(plan, kind), "zero_plan_set_reduce_kernel")


def zero_step(plan: int, grads, master, m, v, params, workspace=None, stream=0) -> None:
    _check(lib().zero_step(plan, _ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                           _ptr(workspace), _ptr(stream)), "zero_step")


def zero_step_qwz(plan: int, grads, master, m, v, params, workspace, bits: int, codes, scales,
                  stream=0) -> None:
    _check(lib().zero_step_qwz(plan, _ptr(grads), _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                               _ptr(workspace), bits, _ptr(codes), _ptr(scales), _ptr(stream)),
           "zero_step_qwz")


def zero_step_pingpong(plan: int, grads, set0, set1, params, stream=0) -> None:
    """set0, set1: (master, m, v) each."""
    (p0, m0, v0), (p1, m1, v1) = set0, set1
    _check(lib().zero_step_pingpong(plan, _ptr(grads), _ptr(p0), _ptr(m0), _ptr(v0), _ptr(p1),
                                    _ptr(m1), _ptr(v1), _ptr(params), _ptr(stream)),
           "zero_step_pingpong")


def zero_plan_state_set(plan: int) -> int:
    s = ctypes.c_int()
    _check(lib().zero_plan_state_set(plan, ctypes.byref(s)), "zero_plan_state_set")
    return s.value


def zero_step_result(plan: int) -> dict:
    sk, lsc, cc = ctypes.c_int(), ctypes.c_float(), ctypes.c_float()
    gn, t = ctypes.c_double(), ctypes.c_int64()
    _check(lib().zero_step_result(plan, ctypes.byref(sk), ctypes.byref(gn), ctypes.byref(cc),
                                  ctypes.byref(lsc), ctypes.byref(t)), "zero_step_result")
    return {"skipped": sk.value, "grad_norm": gn.value, "clip_coef": cc.value,
            "loss_scale": lsc.value, "t": t.value}


def zero_step_overflow(plan: int) -> int:
    o = ctypes.c_int()
    _check(lib().zero_step_overflow(plan, ctypes.byref(o)), "zero_step_overflow")
    return o.value


def zero_gather_layer(plan: int, unit: int, shard_ptrs: Sequence, out, stream=0) -> None:
    arr = (ctypes.c_void_p * max(1, len(shard_ptrs)))(*[_ptr(p) for p in shard_ptrs])
    _check(lib().zero_gather_layer(plan, unit, ctypes.addressof(arr), _ptr(out), _ptr(stream)),
           "zero_gather_layer")


def zero_plan_set_bucket(plan: int, bucket_elems: int) -> int:
    """Turn bucketed steps on (bucket_elems > 0) or off; returns workspace bytes."""
    w = ctypes.c_uint64()
    _check(lib().zero_plan_set_bucket(plan, bucket_elems, ctypes.byref(w)), "zero_plan_set_bucket")
    return w.value


def zero_step_bucket(plan: int, bucket: int, bucket_grads, workspace, stream=0) -> None:
    _check(lib().zero_step_bucket(plan, bucket, _ptr(bucket_grads), _ptr(workspace), _ptr(stream)),
           "zero_step_bucket")


def zero_step_apply(plan: int, master, m, v, params, workspace, stream=0) -> None:
    _check(lib().zero_step_apply(plan, _ptr(master), _ptr(m), _ptr(v), _ptr(params),
                                 _ptr(workspace), _ptr(stream)), "zero_step_apply")


def zero_checkpoint_save(plan: int, directory: str, rank: int, master, m, v, params,
                         flags: int = 0, stream=0) -> None:
    """rank -1: every rank (stages 0-2).  Synchronous."""
    _check(lib().zero_checkpoint_save(plan, os.fsencode(directory), rank, _ptr(master), _ptr(m),
                                      _ptr(v), _ptr(params), flags, _ptr(stream)),
           "zero_checkpoint_save")


def zero_checkpoint_load(plan: int, directory: str, rank: int, master, m, v, params,
                         stream=0) -> None:
    """rank -1: every rank (stages 0-2).  Synchronous."""
    _check(lib().zero_checkpoint_load(plan, os.fsencode(directory), rank, _ptr(master), _ptr(m),
                                      _ptr(v), _ptr(params), _ptr(stream)),
           "zero_checkpoint_load")


def zero_offload_step(plan: int, grads, master, m, v, params, workspace, nthreads: int = 0,
                      stream=0) -> None:
    """master, m, v: host arrays (numpy float32 or CPU tensors); the rest device."""
    _check(lib().zero_offload_step(plan, _ptr(grads), _hptr(master), _hptr(m), _hptr(v),
                                   _ptr(params), _ptr(workspace), nthreads, _ptr(stream)),
           "zero_offload_step")


def zero_cpu_adam(grads16, dtype: int, n: int, loss_scale: float, clip_coef: float, bc1: float,
                  bc2: float, hp, master, m, v, params16, nthreads: int = 0) -> None:
    """Host arrays throughout (numpy or CPU tensors)."""
    _check(lib().zero_cpu_adam(_hptr(grads16), dtype, n, loss_scale, clip_coef, bc1, bc2,
                               ctypes.byref(hp), _hptr(master), _hptr(m), _hptr(v),
                               _hptr(params16), nthreads), "zero_cpu_adam")


def zero_quantize_shard(dtype: int, shard, n: int, bits: int, codes, scales, stream=0) -> None:
    _check(lib().zero_quantize_shard(dtype, _ptr(shard), n, bits, _ptr(codes), _ptr(scales),
                                     _ptr(stream)), "zero_quantize_shard")


def zero_gather_layer_q(plan: int, unit: int, bits: int, code_ptrs: Sequence,
                        scale_ptrs: Sequence, out, stream=0) -> None:
    c = (ctypes.c_void_p * max(1, len(code_ptrs)))(*[_ptr(p) for p in code_ptrs])
    s = (ctypes.c_void_p * max(1, len(scale_ptrs)))(*[_ptr(p) for p in scale_ptrs])
    _check(lib().zero_gather_layer_q(plan, unit, bits, ctypes.addressof(c), ctypes.addressof(s),
                                     _ptr(out), _ptr(stream)), "zero_gather_layer_q")


def zero_state_bytes(psi: int, nd: int, stage: int, K: int = 12) -> int:
    return lib().zero_state_bytes(psi, nd, stage, K)


def zero_comm_volume(psi: int, nd: int, stage: int, exact: int = 0) -> int:
    return lib().zero_comm_volume(psi, nd, stage, exact)


def zero_max_params(mem_bytes: int, nd: int, stage: int, K: int = 12) -> int:
    return lib().zero_max_params(mem_bytes, nd, stage, K)


def zero_plan_profile(plan: int, enable: int) -> None:
    _check(lib().zero_plan_profile(plan, enable), "zero_plan_profile")


def zero_plan_kernel_times(plan: int) -> dict:
    a, b = ctypes.c_double(), ctypes.c_double()
    s, n = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zero_plan_kernel_times(plan, ctypes.byref(a), ctypes.byref(b), ctypes.byref(s),
                                        ctypes.byref(n)), "zero_plan_kernel_times")
    return {"reduce_ms": a.value, "update_ms": b.value, "steps": s.value, "launches": n.value}


def zero_grad_norm_noalloc(grads, nd: int, n: int, rank_stride: int, dtype: int,
                           loss_scale: float, norm_out, overflow_out, stream=0) -> None:
    """Global gradient norm and overflow flag without any allocation: for callers
    that may not allocate device memory.  norm_out (one float64) and overflow_out
    (one int32) are device buffers the caller owns; results land there
    asynchronously on ``stream``."""
    _check(lib().zero_grad_norm_noalloc(_ptr(grads), nd, n, rank_stride, dtype, loss_scale,
                                        _ptr(norm_out), _ptr(overflow_out), _ptr(stream)),
           "zero_grad_norm_noalloc")


def psi_of(shapes: Sequence[Sequence[int]]) -> int:
    return sum(math.prod(s) for s in shapes)
