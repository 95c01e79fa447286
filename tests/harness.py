"""Parity harness: the same seeded inputs through the CPU oracle and through the
CUDA library's C ABI, and the comparison rules.

Tolerances (GPU vs oracle):
  reduced gradient, overflow flags, skip decisions, t, loss scale: bit-exact
  fp32 master, m, v: relative error <= 1e-6, with rel(a, b) = 0 when a and b
      are the same bits, else |a - b| / max(|a|, |b|)
  16-bit parameters: <= 1 unit in the last place (ordered-integer distance)
  grad norm: relative error <= 1e-5
  clip coefficient: within CLIP_ULPS units in the last place of the oracle's

The clip coefficient c = tau / norm is the one value two correct
implementations may round differently: the GPU sums the squares in another
order, and a norm that agrees to 1e-9 can still put c on the other side of a
binary32 rounding boundary.  A coefficient one unit in the last place away
changes the update enough to move a master weight that nearly cancels by far
more than the state tolerance (m = beta1 m + (1 - beta1) g c can cancel to
almost nothing).  So several results are correct: one per admissible c.  The
oracle runs decide which is unique given c: when the GPU reports a c other than
the oracle's own, the oracle checks that it lies within CLIP_ULPS of its own
(CLIP_ULPS covers the GPU norm's worst-case error, 8 * 2^-24 relative) and
takes its step with that admissible c; the state must then be the oracle's
for that c.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

import gen
import oracle

REL_STATE = 1e-6
REL_NORM = 1e-5
ULP_PARAM = 1
CLIP_ULPS = 8


# ---------------------------------------------------------------- comparisons
def rel_err(a: np.ndarray, b: np.ndarray) -> float:
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    if a.size == 0:
        return 0.0
    same = (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    den = np.maximum(np.abs(a64), np.abs(b64))
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.abs(a64 - b64) / np.where(den == 0, 1.0, den)
    r = np.where(same, 0.0, r)
    r = np.where(np.isnan(r), np.inf, r)
    return float(r.max())


def ulp16(a: np.ndarray, b: np.ndarray, skip: Optional[np.ndarray] = None) -> int:
    """Largest ordered-integer distance of two 16-bit arrays, ignoring the
    positions where `skip` is set."""
    def key(x):
        x = np.asarray(x, np.uint16).astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    if np.asarray(a).size == 0:
        return 0
    d = np.abs(key(a) - key(b))
    if skip is not None:
        d = np.where(skip, 0, d)
    return int(d.max())


def ulps32(a: float, b: float) -> int:
    """Distance of two binary32 values in units in the last place (ordered
    integers)."""
    def key(x):
        u = int(np.float32(x).view(np.uint32))
        return -(u & 0x7FFFFFFF) if u & 0x80000000 else u
    return abs(key(a) - key(b))


def admit_clip(c_oracle: float, gpu_result: Optional[dict], what="") -> float:
    """The clip coefficient the oracle's step takes: its own, or the GPU's when
    that one lies within CLIP_ULPS of it (see the module docstring)."""
    if gpu_result is None:
        return c_oracle
    cg = float(np.float32(gpu_result["clip_coef"]))
    if cg == c_oracle:
        return c_oracle
    d = ulps32(cg, c_oracle)
    assert d <= CLIP_ULPS, f"{what}: clip coefficient {cg} is {d} ulp from the oracle's {c_oracle}"
    return cg


def oracle_step_admitting(nd, dtype, g16, master, m, v, params, opt, st,
                          gpu_result: Optional[dict] = None, offload=False, what="") -> dict:
    """One oracle step composed from the oracle's stage functions exactly as its
    zo_step (offload: zo_step_offload) composes them -- reduce, norm, clip
    coefficient, bookkeeping, Adam -- with the clip coefficient admitted by
    admit_clip.  Updates the state in place; returns the oracle's own results."""
    g16 = np.ascontiguousarray(g16, dtype=np.uint16)
    if offload:
        _, g, ovf = oracle.reduce16(nd, dtype, g16, loss_scale=st.loss_scale)
    else:
        g, ovf = oracle.reduce(nd, dtype, g16, loss_scale=st.loss_scale)
    norm = float(np.sqrt(oracle.sumsq(g)))
    c_o = oracle.clip_coef(norm, opt.clip_norm)
    res = oracle.advance(opt, st, ovf)
    if not res.skipped:
        c = admit_clip(c_o, gpu_result, what)
        oracle.adam(g, c, master, m, v, params, dtype, opt, res.bc1, res.bc2)
    out = res.as_dict()
    out["grad_norm"], out["clip_coef"] = norm, c_o
    return out


def assert_state_close(gpu, ora, what=""):
    """Master, m, v within REL_STATE and the 16-bit parameters within ULP_PARAM.
    A NaN is a NaN on both sides whatever its payload (IEEE 754 does not fix the
    payload an operation produces); the 16-bit parameter of an element whose
    master is NaN on both sides is the rounding of a NaN, so it is not compared."""
    for name, x, y in zip(("master", "m", "v"), gpu[:3], ora[:3]):
        e = rel_err(x, y)
        assert e <= REL_STATE, f"{what} {name}: max rel err {e:.3g}"
    both_nan = np.isnan(np.asarray(gpu[0], np.float32)) & np.isnan(np.asarray(ora[0], np.float32))
    u = ulp16(gpu[3], ora[3], skip=both_nan)
    assert u <= ULP_PARAM, f"{what} params: {u} ulp"


# ------------------------------------------------------------------ inputs
@dataclasses.dataclass
class Case:
    shapes: list
    nd: int
    stage: int = 2
    dtype: int = gen.BF16
    grad_sigma: float = 1e-2
    loss_scale: float = 1.0
    dynamic_scale: int = 0
    clip: float = 0.0
    lr: float = 1e-3
    weight_decay: float = 0.0
    decoupled_wd: int = 1
    steps: int = 2
    inf_steps: tuple = ()
    nan_steps: tuple = ()
    units: Optional[List[int]] = None
    seed: int = 0
    growth_interval: int = 1000
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    skip_on_overflow: int = 0

    @property
    def psi(self):
        return int(sum(int(np.prod(s)) for s in self.shapes))

    def opt(self):
        return oracle.Opt(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                          weight_decay=self.weight_decay,
                          decoupled_wd=self.decoupled_wd, clip_norm=self.clip,
                          dynamic_scale=self.dynamic_scale, backoff=0.5,
                          growth_interval=self.growth_interval,
                          skip_on_overflow=self.skip_on_overflow)

    def hparams(self, z):
        return z.hparams(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                         weight_decay=self.weight_decay,
                         decoupled_wd=self.decoupled_wd, clip_norm=self.clip,
                         loss_scale=self.loss_scale, dynamic_scale=self.dynamic_scale,
                         backoff=0.5, growth_interval=self.growth_interval,
                         skip_on_overflow=self.skip_on_overflow)


def from_workload(w, **over) -> Case:
    c = Case(shapes=list(w.shapes), nd=w.nd, stage=w.stage, dtype=w.dtype,
             grad_sigma=w.grad_sigma, loss_scale=w.loss_scale, dynamic_scale=w.dynamic_scale,
             clip=w.clip, lr=w.lr, weight_decay=w.weight_decay, decoupled_wd=w.decoupled_wd,
             steps=w.steps, inf_steps=tuple(w.inf_steps), units=w.units, seed=w.seed)
    return dataclasses.replace(c, **over)


def grads_for_step(c: Case, step: int, n: int, rank_stride: int, scale: float,
                   valid_mask: Optional[np.ndarray] = None) -> np.ndarray:
    """[nd][rank_stride] 16-bit gradients of step `step` (1-based), generated with
    the loss scale in force; +inf / NaN planted on the overflow steps."""
    g = gen.ranks_16_mt(c.seed, gen.STREAM_GRAD, step, c.nd, n, c.grad_sigma, scale, c.dtype,
                        rank_stride=rank_stride)
    if valid_mask is not None:
        g[:, :n][:, ~valid_mask] = 0
    for steps, bits in ((c.inf_steps, 0x7C00 if c.dtype == gen.FP16 else 0x7F80),
                        (c.nan_steps, 0x7E00 if c.dtype == gen.FP16 else 0x7FC0)):
        if step in steps:
            r, i = gen.inf_site(c.seed, step, n, c.nd)
            if valid_mask is not None:
                i = int(np.flatnonzero(valid_mask)[i % int(valid_mask.sum())])
            g[r, i] = bits
    return g


# ------------------------------------------------------------------- runs
@dataclasses.dataclass
class Run:
    master: np.ndarray
    m: np.ndarray
    v: np.ndarray
    params: np.ndarray
    results: list
    g32: Optional[np.ndarray] = None


def stage3_valid_mask(z, plan, nd, rank=0):
    """positions of one rank's shard that hold real (not padding) elements"""
    _, total, nunits, _ = z.zero_plan_layout(plan)
    mask = np.zeros(total, bool)
    for u in range(nunits):
        ln, sl, off = z.zero_plan_unit(plan, u)
        valid = max(0, min(sl, ln - rank * sl))
        mask[off:off + valid] = True
    return mask


def run_gpu(z, c: Case, keep_g32=False, plan_out=None, reduce_kernel=0,
            grads_on_host=False) -> Run:
    """The case through zero_step.  grads_on_host: the ranks' gradients stay in
    page-locked host memory (cudaHostAlloc, mapped into the device's address
    space) and the step reads them there."""
    import torch
    dev = torch.device("cuda", 0)
    plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z),
                              units=c.units if c.stage == 3 else None)
    try:
        if reduce_kernel:
            z.zero_plan_set_reduce_kernel(plan, reduce_kernel)
        shard, padded, nunits, ws = z.zero_plan_layout(plan)
        n = c.psi if c.stage <= 2 else padded
        mask = stage3_valid_mask(z, plan, c.nd) if c.stage == 3 else None
        master0 = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, n, 0.02)
        if mask is not None:
            master0[~mask] = 0
        master = torch.zeros(padded, dtype=torch.float32, device=dev)
        master[:n] = torch.from_numpy(master0).to(dev)
        m = torch.zeros(padded, dtype=torch.float32, device=dev)
        v = torch.zeros(padded, dtype=torch.float32, device=dev)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev) if ws else None
        if grads_on_host:
            grads = torch.empty((c.nd, padded), dtype=torch.int16, pin_memory=True)
        else:
            grads = torch.empty((c.nd, padded), dtype=torch.int16, device=dev)
        stream = torch.cuda.current_stream().cuda_stream
        results = []
        scale = c.loss_scale
        for step in range(1, c.steps + 1):
            g = grads_for_step(c, step, n, padded, scale, mask)
            grads.copy_(torch.from_numpy(g.view(np.int16)))
            z.zero_step(plan, grads, master, m, v, params, work, stream)
            r = z.zero_step_result(plan)
            r["overflow"] = z.zero_step_overflow(plan)
            results.append(r)
            scale = r["loss_scale"]
        torch.cuda.synchronize()
        out = Run(master[:n].cpu().numpy(), m[:n].cpu().numpy(), v[:n].cpu().numpy(),
                  params[:n].cpu().numpy().view(np.uint16), results)
        if keep_g32 and work is not None:
            out.g32 = work[:n].cpu().numpy()
        if plan_out is not None:
            plan_out.append(plan)
            plan = None
        return out
    finally:
        if plan is not None:
            z.zero_plan_destroy(plan)


def run_oracle(c: Case, n: int, padded: int, mask=None, sharded_threads=0,
               follow: Optional[list] = None) -> Run:
    """The oracle over the case's steps.  follow: the GPU's per-step results;
    each step then admits the GPU's clip coefficient (admit_clip)."""
    master = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, n, 0.02)
    if mask is not None:
        master[~mask] = 0
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    st = oracle.new_scalars(c.loss_scale)
    opt = c.opt()
    results = []
    for step in range(1, c.steps + 1):
        g = grads_for_step(c, step, n, padded, st.loss_scale, mask)
        g = np.ascontiguousarray(g[:, :n])
        if follow is not None:
            r = oracle_step_admitting(c.nd, c.dtype, g, master, m, v, params, opt, st,
                                      follow[step - 1], what=f"step {step}")
        elif sharded_threads:
            r = oracle.step_sharded(c.nd, c.dtype, g, master, m, v, params, opt, st,
                                    nthreads=sharded_threads)
        else:
            r = oracle.step(c.nd, c.dtype, g, master, m, v, params, opt, st)
        r["loss_scale"] = st.loss_scale
        r["t"] = st.t
        results.append(r)
    return Run(master, m, v, params, results)


def assert_state_equal(gpu: Run, ora: Run, what=""):
    """Master, m, v and parameters bit for bit (a NaN equals a NaN; the 16-bit
    parameter of an element whose master is NaN on both sides is not compared)."""
    for name, a, b in (("master", gpu.master, ora.master), ("m", gpu.m, ora.m),
                       ("v", gpu.v, ora.v)):
        keep = ~(np.isnan(a) & np.isnan(b))
        assert np.array_equal(a[keep].view(np.uint32), b[keep].view(np.uint32)), f"{what} {name}"
    keep = ~(np.isnan(gpu.master) & np.isnan(ora.master))
    assert np.array_equal(gpu.params[keep], ora.params[keep]), f"{what} params"


def compare_runs(gpu: Run, ora: Run, what=""):
    assert len(gpu.results) == len(ora.results)
    for k, (a, b) in enumerate(zip(gpu.results, ora.results), start=1):
        assert a["skipped"] == b["skipped"], f"{what} step {k}: skip {a} vs {b}"
        assert a["overflow"] == b["overflow"], f"{what} step {k}: overflow {a} vs {b}"
        assert a["t"] == b["t"] and a["loss_scale"] == b["loss_scale"], f"{what} step {k}"
        if np.isfinite(b["grad_norm"]):
            e = abs(a["grad_norm"] - b["grad_norm"]) / max(abs(b["grad_norm"]), 1e-300)
            assert e <= REL_NORM, f"{what} step {k}: norm {a['grad_norm']} vs {b['grad_norm']}"
            if not a["skipped"]:
                d = ulps32(a["clip_coef"], b["clip_coef"])
                assert d <= CLIP_ULPS, f"{what} step {k}: clip {a['clip_coef']} vs {b['clip_coef']}"
        else:
            assert not np.isfinite(a["grad_norm"])
    assert_state_close((gpu.master, gpu.m, gpu.v, gpu.params),
                       (ora.master, ora.m, ora.v, ora.params), what)


# ------------------------------------------------------- full-size helpers
def oracle_norm_streamed(seed, step, nd, n, sigma, scale, dtype, inf_at=None, nthreads=None,
                         chunk=1 << 21, index_map=None):
    """The oracle's global norm and overflow flag over n elements whose gradients
    are too many to hold at once: the flat vector is cut into contiguous ranges
    (one per host thread, like ranks of the sharded oracle), each range streamed
    in chunks through oracle.reduce / oracle.sumsq, and the range partials added
    in range order.  inf_at = (rank, index) plants +inf there."""
    import concurrent.futures
    import os
    nthreads = nthreads or min(os.cpu_count() or 1, 32)
    bounds = [n * k // nthreads for k in range(nthreads + 1)]
    inf_bits = 0x7C00 if dtype == gen.FP16 else 0x7F80

    def work(k):
        lo, hi = bounds[k], bounds[k + 1]
        part, ovf = 0.0, False
        for a in range(lo, hi, chunk):
            b = min(a + chunk, hi)
            g16 = gen.ranks_16(seed, gen.STREAM_GRAD, step, nd, b - a, sigma, scale, dtype,
                               index0=a)
            if inf_at is not None and a <= inf_at[1] < b:
                g16[inf_at[0], inf_at[1] - a] = inf_bits
            g, o = oracle.reduce(nd, dtype, g16, loss_scale=scale)
            ovf = ovf or o
            part = part + oracle.sumsq(g)
        return part, ovf

    with concurrent.futures.ThreadPoolExecutor(nthreads) as ex:
        parts = list(ex.map(work, range(nthreads)))
    total = 0.0
    ovf = False
    for p, o in parts:
        total = total + p
        ovf = ovf or o
    return float(np.sqrt(total)), ovf


def sample_indices(n, shard, nd, k=1 << 16, seed=1):
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, n, k).tolist())
    for r in range(nd + 1):
        for d in (-1, 0, 1):
            j = r * shard + d
            if 0 <= j < n:
                idx.add(j)
    idx.update(range(max(0, n - 9), n))
    idx.update(range(min(n, 9)))
    return np.array(sorted(idx), np.int64)


def oracle_sampled_grads(seed, step, nd, idx, sigma, scale, dtype, inf_at=None):
    g16 = np.stack([gen.s16_at(seed, gen.STREAM_GRAD, step, r, idx, sigma, scale, dtype)
                    for r in range(nd)])
    if inf_at is not None:
        hit = np.flatnonzero(idx == inf_at[1])
        if hit.size:
            g16[inf_at[0], hit[0]] = 0x7C00 if dtype == gen.FP16 else 0x7F80
    return g16
