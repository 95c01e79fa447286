#!/usr/bin/env python3
"""Benchmark of the ZeRO-DP sharded mixed-precision optimizer step on GB300.

Workload: the GPT-2 1.5B parameter list (48 layers, h 1600, ffn 6400, vocab
50257, ctx 1024: 1,557,611,200 parameters), Nd = 16 emulated data-parallel
ranks, ZeRO-2, fp16 gradients N(0, 1e-3) x 65536 under dynamic loss scaling,
clip by global norm 1.0, Adam (lr 1e-3, betas 0.9/0.999, eps 1e-8).  Synthetic
seeded inputs; no weights or data.

One step = one zero_step call: the 16-way fixed-order reduce-scatter and
average, unscale + overflow flag, global norm, clip, Adam on the fp32 master,
m and v, the fp16 cast and the write-back of every shard into the flat
parameter buffer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  For N > 1 (torchrun), every rank runs its own
independent replica of the workload on its own GPU (the path has no data
exchange between GPUs here): weak scaling, barrier + max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sharded Adam step params/s and HBM GB/s vs GB300 peak (GPT-2 1.5B, Nd=16)"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
STATUS_BYTES = 72            # the optimizer scalars + step status zero_step_result copies


# --------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def dist_init(backend: str):
    import torch.distributed as dist
    rank, local, ws = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return rank, local, ws


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_scalar(x: float, op: str, device=None) -> float:
    """max or sum of one float over ranks (timing bookkeeping only)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ("zero_common.cuh", "zero_step_kernels.cuh", "zero_step_table.cuh",
                  "zero_step_fp16.cu", "zero_step_bf16.cu", "zero_tma.cuh", "zero_qwz.cuh")


def kernel_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(f.encode())
        with open(os.path.join(ROOT, "zero_sharded_mixed_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(kernel: str, psi: int, nd: int):
    """DRAM bytes per launch of `kernel` on this workload, scaled from the committed ncu
    capture in profiles/dram_traffic.txt; None if the kernels changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        sha = kernel_source_sha()
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) < 6 or parts[0].startswith("#") or parts[0] != kernel:
                    continue
                if parts[1] != sha or int(parts[3]) != nd:
                    continue
                return (int(parts[4]) + int(parts[5])) * psi / int(parts[2])
    except (OSError, ValueError):
        pass
    return None


def host_mem_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def host_device_pointer(ptr: int):
    """The device address of page-locked host memory at ptr (cudaHostGetDevicePointer,
    through the CUDA runtime this process loaded), or None where it is not mapped."""
    import ctypes
    lib = None
    try:
        with open("/proc/self/maps") as f:
            for line in f:
                if "libcudart" in line:
                    lib = line.split()[-1]
                    break
    except OSError:
        return None
    if lib is None:
        return None
    try:
        rt = ctypes.CDLL(lib)
        d = ctypes.c_void_p()
        rc = rt.cudaHostGetDevicePointer(ctypes.byref(d), ctypes.c_void_p(ptr), 0)
    except (OSError, AttributeError):
        return None
    return d.value if rc == 0 and d.value else None


class HugePinned:
    """nbytes of page-locked host memory backed by transparent huge pages:
    anonymous pages with MADV_HUGEPAGE, page-locked by cudaHostRegister (which
    faults them in).  On these hosts a ~50 GB cudaHostAlloc buffer copied to the
    GPU at 115-207 GB/s, depending on the run and on how the copy was cut; this
    one copies at the link's 211 GB/s whole or in chunks."""

    def __init__(self, nbytes: int):
        import mmap
        import numpy as np
        import torch
        self.nbytes = nbytes
        self.map = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        try:
            self.map.madvise(mmap.MADV_HUGEPAGE)
        except (AttributeError, OSError):
            pass
        view = np.frombuffer(self.map, dtype=np.uint8)
        self.ptr = view.ctypes.data
        del view
        self.registered = False
        rc = torch.cuda.cudart().cudaHostRegister(self.ptr, nbytes, 0)
        if int(rc) != 0:
            self.map.close()
            raise RuntimeError(f"cudaHostRegister failed ({int(rc)})")
        self.registered = True

    def huge_fraction(self) -> float:
        """Share of the mapping backed by transparent huge pages (AnonHugePages of
        its /proc/self/smaps entry): on a host whose memory is fragmented the kernel
        falls back to 4 KB pages, which the GPU copies from far more slowly."""
        lo, hi = self.ptr, self.ptr + self.nbytes
        try:
            with open("/proc/self/smaps") as f:
                inside, huge = False, 0
                for line in f:
                    head = line.split()[0]
                    if "-" in head and not head.endswith(":"):
                        a, b = (int(x, 16) for x in head.split("-"))
                        inside = a < hi and b > lo
                    elif inside and head == "AnonHugePages:":
                        huge += int(line.split()[1]) * 1024
            return huge / self.nbytes
        except (OSError, ValueError):
            return 0.0

    def tensor(self, dtype, shape):
        import torch
        return torch.frombuffer(self.map, dtype=dtype).view(shape)

    def release(self):
        """Unregister and unmap; call after the device is done with the memory and
        no tensor made by tensor() is left."""
        import gc
        import torch
        if self.registered:
            torch.cuda.cudart().cudaHostUnregister(self.ptr)
            self.registered = False
        gc.collect()
        try:
            self.map.close()
        except BufferError:          # a view is still alive: the mapping goes with it
            pass


def huge_host_array(n: int, dtype):
    """A host numpy array of n elements in anonymous memory advised to use
    transparent huge pages (MADV_HUGEPAGE), zero-filled: host state arrays of tens
    of GB otherwise sit on small pages.  The mapping lives as long as the array."""
    import mmap
    import numpy as np
    nbytes = max(1, n * np.dtype(dtype).itemsize)
    mp = mmap.mmap(-1, nbytes, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    try:
        mp.madvise(mmap.MADV_HUGEPAGE)
    except (AttributeError, OSError):
        pass
    return np.frombuffer(mp, dtype=dtype, count=n)


def pinning_fits(nbytes: int, device=None, avail=None):
    """Whether every rank on this node can pin nbytes of host memory at once.
    MemAvailable must cover LOCAL_WORLD_SIZE such buffers plus 8 GB each; the
    ranks decide together (one rank short and all skip), so they all take the
    same path through the collectives that follow.  Returns (fits, avail, need)."""
    _, _, ws = dist_env()
    local_ws = int(os.environ.get("LOCAL_WORLD_SIZE", str(ws)))
    avail = host_mem_available() if avail is None else avail
    need = local_ws * (nbytes + (8 << 30))
    short = reduce_scalar(0.0 if avail >= need else 1.0, "max", device)
    return short == 0.0, avail, need


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of the SM clock and throttle reasons."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        if not rows:
            return None
        t0, t1 = self.window if self.window else (rows[0][0], rows[-1][0])
        inside = [p for ts, p in rows if t0 - 0.25 <= ts <= t1 + 0.25] or [p for _, p in rows]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(p[2]) for p in inside if not math.isnan(num(p[2]))]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for p in inside:
            for name, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][3]), "reasons": sorted(reasons),
                "samples": len(inside),
                "power_w_max": max((num(p[4]) for p in inside), default=None)}


# ----------------------------------------------------------------- workload
WORKLOADS = ("gpt2-1.5b", "gpt2-small", "tiny", "llama3-8b")


def metric_of(w):
    if w.name == "gpt2-1.5b":
        return METRIC
    return f"sharded Adam step params/s and HBM GB/s vs GB300 peak ({w.name}, Nd={w.nd})"


def workload(psi=None, name="gpt2-1.5b", nd=None):
    """The GPT-2 1.5B workload (default) or another named one; with psi, a flat
    single-tensor model of psi parameters under the same settings (small cases
    for profiling), with nd ranks when nd is given."""
    import dataclasses
    from gen import workloads
    w = {"gpt2-1.5b": workloads.gpt2_xl, "gpt2-small": workloads.gpt2_small,
         "tiny": workloads.tiny, "llama3-8b": workloads.llama3_8b}[name]()
    if psi:
        w = dataclasses.replace(w, name=f"flat-{psi}", shapes=[(psi,)])
    if nd:
        w = dataclasses.replace(w, nd=nd)
    return w


DESCRIPTIONS = {
    "gpt2-1.5b": "GPT-2 1.5B parameter list (48 layers, h=1600, ffn=6400, vocab 50257, ctx 1024)",
    "gpt2-small": "GPT-2 small parameter list (12 layers, h=768, ffn=3072, vocab 50257, ctx 1024)",
    "tiny-flat-4t": "tiny flat model: 4 tensors [512x1024, 1024, 1024x512, 512]",
    "llama3-8b": "LLaMA-3-8B parameter list (32 layers, h=4096, ffn=14336, 32q/8kv, vocab 128256)",
}


def config_of(w, padded):
    desc = (f"{w.name}: {DESCRIPTIONS.get(w.name, w.name)}, {len(w.shapes)} tensors"
            if len(w.shapes) > 1 else
            f"{w.name}: one flat tensor of {w.psi} parameters, {w.nd} ranks")
    return {"workload": desc,
            "psi": w.psi, "nd": w.nd, "zero_stage": w.stage, "padded_elems": padded,
            "grads": (f"{'fp16' if w.dtype == 0 else 'bf16'} N(0,{w.grad_sigma:g})"
                      + (f" x {w.loss_scale:g} loss scale" if w.loss_scale != 1 else "")
                      + (" (dynamic)" if w.dynamic_scale else "")),
            "clip_norm": w.clip,
            "optimizer": (f"{'AdamW' if w.weight_decay else 'Adam'} lr {w.lr:g} betas "
                          f"({w.beta1:g}, {w.beta2:g}) eps {w.eps:g}"
                          + (f" wd {w.weight_decay:g}" if w.weight_decay else "")),
            "l2": (f"inputs ({(2 * w.nd + 14) * padded / 1e9:.2f} GB resident) vs the 129 MB L2"
                   + ("; larger, no flush needed" if (2 * w.nd + 14) * padded > (1 << 30) else
                      "; L2 flushed between steps (256 MB written, then 256 MB read)")),
            "parallelism": "Nd ranks emulated in one GPU's HBM"}


# ----------------------------------------------------------- CPU baseline
def oracle_sample(w, n_sample: int, threads: int, repeats_min_s: float = 0.0, max_repeats=1):
    """Time the oracle (as it stands) on the first n_sample elements of the flat
    vector with all Nd ranks' contributions; returns (params/s, seconds/step, reps)."""
    import numpy as np
    import gen
    import oracle
    g = gen.ranks_16(w.seed, gen.STREAM_GRAD, 1, w.nd, n_sample, w.grad_sigma, w.loss_scale,
                     w.dtype)
    master0 = gen.f32(w.seed, gen.STREAM_MASTER, 0, 0, n_sample, w.master_sigma)
    opt = oracle.Opt(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                     weight_decay=w.weight_decay, decoupled_wd=w.decoupled_wd,
                     clip_norm=w.clip, dynamic_scale=w.dynamic_scale, backoff=0.5,
                     growth_interval=1000)
    master, m, v = master0.copy(), np.zeros(n_sample, np.float32), np.zeros(n_sample, np.float32)
    params = np.zeros(n_sample, np.uint16)
    st = oracle.new_scalars(w.loss_scale)
    shard = oracle.shard_elems(n_sample, w.nd)
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.step_sharded(w.nd, w.dtype, g, master, m, v, params, opt, st, shard=shard,
                            nthreads=threads)
        times.append(time.perf_counter() - t0)
        if len(times) >= max_repeats or time.perf_counter() - t_start >= repeats_min_s:
            break
    per_step = sum(times) / len(times)
    return n_sample / per_step, per_step, len(times)


def oracle_threads(nd: int) -> int:
    return max(1, min(os.cpu_count() or 1, nd))


# ------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild

    rank, local, ws = dist_init("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    zbuild.build()
    w = workload(args.psi, args.workload, args.nd)
    hp = z.hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                   decoupled_wd=w.decoupled_wd, clip_norm=w.clip, loss_scale=w.loss_scale,
                   dynamic_scale=w.dynamic_scale, backoff=0.5, growth_interval=1000)
    plan = z.zero_plan_create(w.psi, w.nd, w.stage, w.dtype, w.shapes, hp)
    if args.reduce_kernel == "tma":
        z.zero_plan_set_reduce_kernel(plan, z.REDUCE_TMA)
    shard, padded, _, ws_bytes = z.zero_plan_layout(plan)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    grads = torch.empty((w.nd, padded), dtype=torch.int16, device=dev)
    master = torch.zeros(padded, dtype=torch.float32, device=dev)
    m = torch.zeros(padded, dtype=torch.float32, device=dev)
    v = torch.zeros(padded, dtype=torch.float32, device=dev)
    params = torch.zeros(padded, dtype=torch.int16, device=dev)
    work = torch.empty(max(ws_bytes, 16) // 4, dtype=torch.float32, device=dev)
    gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, 1, w.nd, w.psi, w.grad_sigma,
                      w.loss_scale, w.dtype, rank_stride=padded, cuda_stream=sp)
    gen.cuda_f32(master.data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, w.psi, w.master_sigma,
                 cuda_stream=sp)
    torch.cuda.synchronize(dev)

    def step():
        z.zero_step(plan, grads, master, m, v, params, work, sp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    warm = z.zero_step_result(plan)

    # ---- device-timed region: K steps, inputs resident in HBM, exactly the
    # launch sequence the library ships (no per-kernel events between the
    # reduce pass and its programmatic dependent) ----
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    z.zero_plan_profile(plan, 0)
    launches0 = z.zero_plan_kernel_times(plan)["launches"]
    small = (2 * w.nd + 14) * padded <= (1 << 30)     # inputs could stay in L2: flush
    flush = l2_flush(torch, dev) if small else None
    barrier(dev)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    ms_local = _timed_steps(torch, stream, step, args.steps, flush)
    t_wall1 = time.time()
    barrier(dev)
    sampler.mark(t_wall0, t_wall1)
    launches1 = z.zero_plan_kernel_times(plan)["launches"]
    ms_total = reduce_scalar(ms_local, "max", dev)

    # ---- a second pass of K steps with the plan's per-kernel events on: the
    # split between the passes and the dominant kernel's time (the events sit
    # between the two kernels, so this pass's step time is reported apart) ----
    z.zero_plan_profile(plan, 1)
    barrier(dev)
    torch.cuda.synchronize(dev)
    ms_prof_local = _timed_steps(torch, stream, step, args.steps, flush)
    barrier(dev)
    kt = z.zero_plan_kernel_times(plan)
    z.zero_plan_profile(plan, 0)
    clocks = sampler.stop()
    ms_prof_total = reduce_scalar(ms_prof_local, "max", dev)
    res = z.zero_step_result(plan)

    psi, nd, K = w.psi, w.nd, args.steps
    ms_step = ms_total / K
    value = psi * K * ws / (ms_total / 1e3)
    peak, peak_kind = measured_peaks()
    roof_bytes = (2 * nd + 26) * psi
    floor_bytes = (2 * nd + 34) * psi
    step_gbs = roof_bytes / (ms_step / 1e3) / 1e9
    launches = launches1 - launches0

    # dominant kernel: the pass with more device time
    a_ms = kt["reduce_ms"] / max(kt["steps"], 1)
    b_ms = kt["update_ms"] / max(kt["steps"], 1)
    if a_ms >= b_ms:
        kname, kms, kbytes = "k_reduce (fold + unscale + flag + norm partials, writes fp32 g)", \
            a_ms, (2 * nd + 4) * psi
        traffic = ncu_traffic("k_reduce", psi, nd)
    else:
        kname, kms, kbytes = "k_update (clip + Adam + cast + write-back)", b_ms, 30 * psi
        traffic = ncu_traffic("k_update", psi, nd)
    achieved = kbytes / (kms / 1e3) / 1e9

    out = {
        "metric": metric_of(w), "value": value, "unit": "params/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; shape list only, no weights)",
        "config": config_of(w, padded),
        "hbm_gbs_roofline_bytes": step_gbs,
        "roofline_bytes_per_elem": 2 * nd + 26,
        "frac_of_measured_hbm": step_gbs / peak,
        "frac_of_nominal_hbm": step_gbs / NOMINAL_HBM_GBS,
        "hbm_gbs_floor_bytes": floor_bytes / (ms_step / 1e3) / 1e9,
        "floor_bytes_per_elem": 2 * nd + 34,
        "kernel_ms": {"reduce": a_ms, "update": b_ms,
                      "source": "a separate pass of the same K steps with per-kernel CUDA events "
                                "on the launching stream",
                      "ms_per_step_with_events": ms_prof_total / K},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind ==
                     "measured" else "fallback", "unit": "GB/s", "frac": achieved / peak,
                     "algorithmic_bytes_per_launch": kbytes, "traffic": traffic,
                     "traffic_source": "ncu dram bytes of a 64M-parameter capture scaled by "
                                       "elements (profiles/dram_traffic.txt)" if traffic else None},
        "reduce_kernel": args.reduce_kernel,
        "gpu_launches": launches,
        "clocks": clocks,
        "step_result": {k: res[k] for k in ("skipped", "grad_norm", "clip_coef", "loss_scale",
                                            "t")},
        "warmup_result": {"t": warm["t"], "grad_norm": warm["grad_norm"]},
    }

    # ---- end to end through the C ABI: host gradients copied in every step ----
    if not args.no_e2e:
        out["e2e"] = e2e_leg(args, z, plan, w, grads, master, m, v, params, work, dev, stream)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only) ----
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        n_s = args.cpu_sample
        thr = oracle_threads(nd)
        pps, per, reps = oracle_sample(w, n_s, thr, repeats_min_s=10.0, max_repeats=50)
        out["cpu_baseline"] = {
            "value": pps, "unit": "params/s", "cores": thr, "kind": "oracle",
            "sample": f"first {n_s} elements of the flat vector x {nd} ranks' fp16 gradients, "
                      f"one full oracle step each ({reps} steps, {per:.3f} s/step)"}

    z.zero_plan_destroy(plan)

    # ---- the other workloads, measured in the same run (rank 0, N = 1 only) ----
    if rank == 0 and ws == 1 and not args.no_other_configs:
        del grads, master, m, v, params, work
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        out["other_configs"] = other_configs(args)

    if rank == 0:
        print(json.dumps(out), flush=True)


def workload_point(w, k: int, pingpong: bool = False) -> dict:
    """One stages 0-2 workload through zero_step: 3 warm-up steps, then k timed
    steps on the device (L2 flushed between steps when the inputs would fit in
    it); step time, params/s and GB/s on the 2Nd + 26 roofline bytes.  pingpong:
    the same steps through zero_step_pingpong too (two state sets, one pass)."""
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    peak, _ = measured_peaks()
    plan = _plan_for(z, w)
    try:
        _, padded, _, ws = z.zero_plan_layout(plan)
        grads = torch.empty((w.nd, padded), dtype=torch.int16, device=dev)
        master = torch.zeros(padded, dtype=torch.float32, device=dev)
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev)
        gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, 1, w.nd, w.psi, w.grad_sigma,
                          w.loss_scale, w.dtype, rank_stride=padded, cuda_stream=sp)
        gen.cuda_f32(master.data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, w.psi, w.master_sigma,
                     cuda_stream=sp)

        def step():
            z.zero_step(plan, grads, master, m, v, params, work, sp)
        for _ in range(3):
            step()
        torch.cuda.synchronize(dev)
        small = (2 * w.nd + 14) * padded <= (1 << 30)
        flush = l2_flush(torch, dev) if small else None
        ms = _timed_steps(torch, stream, step, k, flush) / k
        roof = (2 * w.nd + 26) * w.psi
        res = {"psi": w.psi, "nd": w.nd, "stage": w.stage, "path": z.zero_plan_path(plan),
               "ms_per_step": ms, "params_per_s": w.psi / (ms / 1e3),
               "hbm_gbs_roofline_bytes": roof / (ms / 1e3) / 1e9,
               "frac_of_measured_hbm": roof / (ms / 1e3) / 1e9 / peak, "steps": k,
               "l2": "flushed between steps" if small else "inputs larger than L2"}
        if pingpong:
            other = [torch.zeros_like(master) for _ in range(3)]

            def step_pp():
                z.zero_step_pingpong(plan, grads, (master, m, v), other, params, sp)
            for _ in range(3):
                step_pp()
            torch.cuda.synchronize(dev)
            ms_pp = _timed_steps(torch, stream, step_pp, k, flush) / k
            res["pingpong"] = {
                "what": "zero_step_pingpong: one pass over two state sets, a skipped step "
                        "rewrites the 16-bit parameters from the current set",
                "ms_per_step": ms_pp, "params_per_s": w.psi / (ms_pp / 1e3),
                "frac_of_measured_hbm": roof / (ms_pp / 1e3) / 1e9 / peak,
                "vs_zero_step": ms / ms_pp}
        return res
    finally:
        z.zero_plan_destroy(plan)
        torch.cuda.empty_cache()


def run_pingpong(args):
    """The named workload with its clip turned off (fp16 dynamic loss scaling
    keeps the skip): zero_step (two passes through an fp32 gradient, since the
    overflow flag must be known before any update) against zero_step_pingpong
    (one pass over two state sets), K device-timed steps each."""
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild
    zbuild.build()
    w = dataclasses.replace(workload(args.psi, args.workload, args.nd), clip=0.0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    peak, _ = measured_peaks()
    plan = _plan_for(z, w)
    try:
        _, padded, _, ws = z.zero_plan_layout(plan)
        grads = torch.empty((w.nd, padded), dtype=torch.int16, device=dev)
        sets = [[torch.zeros(padded, dtype=torch.float32, device=dev) for _ in range(3)]
                for _ in range(2)]
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev)
        gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, 1, w.nd, w.psi, w.grad_sigma,
                          w.loss_scale, w.dtype, rank_stride=padded, cuda_stream=sp)
        gen.cuda_f32(sets[0][0].data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, w.psi,
                     w.master_sigma, cuda_stream=sp)
        K = args.steps
        small = (2 * w.nd + 14) * padded <= (1 << 30)
        flush = l2_flush(torch, dev) if small else None

        def two_pass():
            z.zero_step(plan, grads, *sets[0], params, work, sp)

        def one_pass():
            z.zero_step_pingpong(plan, grads, sets[0], sets[1], params, sp)
        for _ in range(max(3, args.warmup)):
            two_pass()
        ms2 = _timed_steps(torch, stream, two_pass, K, flush) / K
        for _ in range(max(3, args.warmup)):
            one_pass()
        ms1 = _timed_steps(torch, stream, one_pass, K, flush) / K
        roof = (2 * w.nd + 26) * w.psi
        print(json.dumps({
            "mode": "pingpong", "workload": f"{w.name} with the clip off", "psi": w.psi,
            "nd": w.nd, "grads": "fp16 dynamic loss scale" if w.dynamic_scale else "static",
            "zero_step_ms": ms2, "zero_step_pingpong_ms": ms1, "speedup": ms2 / ms1,
            "roofline_bytes_per_elem": 2 * w.nd + 26,
            "frac_of_measured_hbm": {"zero_step": roof / (ms2 / 1e3) / 1e9 / peak,
                                     "zero_step_pingpong": roof / (ms1 / 1e3) / 1e9 / peak},
            "steps": K, "t": z.zero_step_result(plan)["t"],
            "state_set": z.zero_plan_state_set(plan)}), flush=True)
    finally:
        z.zero_plan_destroy(plan)


def other_configs(args) -> dict:
    """The other workloads of the benchmark's configuration list, each timed on the
    device in this run: the tiny flat model, GPT-2 small, LLaMA-3-8B ZeRO-3 (the
    resident shard's update, the 34 unit gathers, and the 4-bit qwZ step), and two
    points of the bandwidth sweep.  A workload that fails is recorded, not fatal."""
    import argparse
    from gen import workloads as W
    res = {}
    jobs = [("tiny-flat-4t", lambda: workload_point(W.tiny(), 200, pingpong=True)),
            ("gpt2-small", lambda: workload_point(W.gpt2_small(), 20)),
            ("llama3-8b", lambda: stage3_measure(argparse.Namespace(
                layers=0, vocab=0, nd=0, qwz=4, warmup=3, steps=10))),
            ("sweep-2^24-nd8", lambda: workload_point(W.sweep(1 << 24, 8), 200)),
            ("sweep-2^28-nd8", lambda: workload_point(W.sweep(1 << 28, 8), 20))]
    for name, fn in jobs:
        try:
            res[name] = fn()
        except Exception as e:                      # noqa: BLE001 -- recorded in the line
            res[name] = {"error": f"{type(e).__name__}: {e}"}
    return res


def e2e_leg(args, z, plan, w, grads, master, m, v, params, work, dev, stream):
    """Same metric through the public API with host-resident gradients: every
    step copies the 16 ranks' fp16 gradients from pinned host memory to the
    device, runs zero_step and reads the step status back."""
    import torch
    nbytes = grads.numel() * 2
    fits, avail, need = pinning_fits(nbytes, dev)
    if not fits:
        return {"value": None, "unit": "params/s", "h2d_bytes_per_step": nbytes,
                "d2h_bytes_per_step": STATUS_BYTES,
                "skipped": f"host has {avail / 1e9:.0f} GB available; pinning every local "
                           f"rank's gradients needs {need / 1e9:.0f} GB"}
    # huge-page memory when the host can back the buffer with huge pages; when its
    # memory is too fragmented for that (measured: 30 GB/s from a 4 KB-page buffer of
    # this size, against 97 GB/s from cudaHostAlloc), the driver's pinned allocation
    pinned, huge = None, 0.0
    try:
        pinned = HugePinned(nbytes)
        huge = pinned.huge_fraction()
        if huge < 0.9:
            pinned.release()
            pinned = None
    except RuntimeError:
        pinned = None
    if pinned is not None:
        host = pinned.tensor(grads.dtype, grads.shape)
        host_kind = (f"transparent-huge-page memory ({100 * huge:.0f}% huge pages) page-locked "
                     "with cudaHostRegister")
    else:
        host = torch.empty(grads.shape, dtype=grads.dtype, pin_memory=True)
        host_kind = (f"cudaHostAlloc (torch pin_memory); huge pages covered {100 * huge:.0f}% "
                     "of a first try")
    host.copy_(grads)
    sp = stream.cuda_stream
    K = max(3, min(args.steps, args.e2e_steps))
    # Two device gradient buffers when they fit: step k+1's gradients are copied on
    # a copy stream while step k runs, and a buffer is refilled only after the step
    # that read it has finished.  Every step still copies its own 49.8 GB and reads
    # its status back; with one buffer the copies and steps alternate.
    two = torch.cuda.mem_get_info(dev)[0] > nbytes + (4 << 30)
    bufs = [grads, torch.empty_like(grads)] if two else [grads]
    cs = torch.cuda.Stream(dev)
    consumed = [None] * len(bufs)
    copied = [None] * len(bufs)

    def h2d(k):
        i = k % len(bufs)
        if consumed[i] is None:                     # first use: after the queued work
            ev = torch.cuda.Event()
            ev.record(stream)
            cs.wait_event(ev)
        else:
            cs.wait_event(consumed[i])
        with torch.cuda.stream(cs):
            for r in range(bufs[i].shape[0]):       # one copy per rank row
                bufs[i][r].copy_(host[r], non_blocking=True)
        copied[i] = torch.cuda.Event()
        copied[i].record(cs)

    def step(k):
        i = k % len(bufs)
        stream.wait_event(copied[i])
        z.zero_step(plan, bufs[i], master, m, v, params, work, sp)
        consumed[i] = torch.cuda.Event()
        consumed[i].record(stream)
        z.zero_step_result(plan)

    def run(n):
        h2d(0)
        for k in range(n):
            if len(bufs) > 1 and k + 1 < n:
                h2d(k + 1)
            step(k)
            if len(bufs) == 1 and k + 1 < n:
                h2d(k + 1)

    # Warm-up: pairs of steps until two consecutive pairs agree within 5 % (at most
    # 30 s).  Right after a large workload the host's background page compaction can
    # slow the link for several seconds (measured: 85 GB/s in the first pass after the
    # GPU test suite, 190 GB/s eight seconds later); the timed steps then see the
    # link's steady rate.
    warm, prev, deadline = 0, None, time.perf_counter() + 30.0
    while True:
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        run(2)
        torch.cuda.synchronize(dev)
        dt = time.perf_counter() - t0
        warm += 2
        if (prev is not None and abs(dt - prev) <= 0.05 * prev) or time.perf_counter() > deadline:
            break
        prev = dt
    # The other way to take host-resident gradients: zero_step reads them in place
    # from the page-locked buffer (its device address from cudaHostGetDevicePointer).
    # Which of the two moves 49.8 GB faster depends on the host's state (measured
    # right after the GPU test suite: in place 204 GB/s against 68 for the copies on
    # one box, 126 against 190 on another), so two warm-up pairs of each decide.
    dptr = host_device_pointer(host.data_ptr())

    def step_in_place():
        z.zero_step(plan, dptr, master, m, v, params, work, sp)
        z.zero_step_result(plan)

    in_place = False
    if dptr is not None:
        for _ in range(2):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            step_in_place()
            step_in_place()
            dt_in = time.perf_counter() - t0
            warm += 2
        in_place = dt_in < 0.95 * dt
    # each rank decides for itself (no collective runs inside the timed steps)
    barrier(dev)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    if in_place:
        for _ in range(K):
            step_in_place()
    else:
        run(K)
    torch.cuda.synchronize(dev)
    dt = reduce_scalar(time.perf_counter() - t0, "max", dev)
    _, _, ws = dist_env()
    del host
    if pinned is not None:
        pinned.release()
    del bufs
    return {"value": w.psi * K * ws / dt, "unit": "params/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": STATUS_BYTES, "steps": K, "warmup_steps": warm,
            "ms_per_step": dt / K * 1e3,
            "h2d_gbs": nbytes / (dt / K) / 1e9,
            "transfer": ("zero_step reads the gradients in place from page-locked host memory"
                         if in_place else "cudaMemcpyAsync per rank row into device buffers"),
            "device_buffers": 0 if in_place else (2 if two else 1),
            "overlap": ("none needed: the reduce pass reads over the host link" if in_place else
                        "step k+1's copy runs during step k" if two else
                        "copies and steps alternate"),
            "host_memory": host_kind}


# ------------------------------------------------------------ sweep and ZeRO-3
def _plan_for(z, w, units=None):
    hp = z.hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                   decoupled_wd=w.decoupled_wd, clip_norm=w.clip, loss_scale=w.loss_scale,
                   dynamic_scale=w.dynamic_scale, backoff=0.5, growth_interval=1000)
    return z.zero_plan_create(w.psi, w.nd, w.stage, w.dtype, w.shapes, hp, units=units)


def l2_flush(torch, dev):
    """An L2 flush for small inputs: write a 256 MB buffer (twice the 129 MB L2),
    then read another one.  The read evicts the written lines, so their write-back
    happens here, outside the timed step, and the step starts with L2 holding only
    clean lines of no use to it."""
    wbuf = torch.empty(1 << 28, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(1 << 26, dtype=torch.float32, device=dev)

    def flush():
        wbuf.fill_(1)
        rbuf.sum()
    return flush


def _timed_steps(torch, stream, step, k, flush=None):
    """Device time of k calls of step(): one event pair around all of them, or,
    with flush (l2_flush) between steps, one event pair per step."""
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(k)]
    for a, b in evs:
        flush()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


def run_sweep(args):
    """Bandwidth sweep: flat bf16 models, psi x nd, ZeRO-2, no clip (the fused
    single pass); m and v from 5 warm-up steps; one JSON line per point."""
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild
    from gen import workloads as W
    zbuild.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    peak, _ = measured_peaks()
    flush = l2_flush(torch, dev)
    for psi in ([args.psi] if args.psi else W.SWEEP_PSI):
        for nd in ([args.nd] if args.nd else W.SWEEP_ND):
            w = W.sweep(psi, nd)
            line = {"mode": "sweep", "metric": "sharded Adam step HBM GB/s, bandwidth sweep",
                    "psi": psi, "nd": nd, "zero_stage": 2, "dtype": "bf16 grads, f32 state"}
            torch.cuda.empty_cache()
            need = (2 * nd + 14) * psi + (1 << 30)
            if need > torch.cuda.mem_get_info()[0]:
                line["skipped"] = f"needs {need / 1e9:.0f} GB"
                print(json.dumps(line), flush=True)
                continue
            plan = _plan_for(z, w)
            shard, padded, _, _ = z.zero_plan_layout(plan)
            grads = torch.empty((nd, padded), dtype=torch.int16, device=dev)
            master = torch.zeros(padded, dtype=torch.float32, device=dev)
            m, v = torch.zeros_like(master), torch.zeros_like(master)
            params = torch.zeros(padded, dtype=torch.int16, device=dev)
            gen.cuda_f32(master.data_ptr(), 0, gen.STREAM_MASTER, 0, 0, psi, 0.02, cuda_stream=sp)
            for step in range(1, 6):                                   # 5 warm-up steps
                gen.cuda_ranks_16(grads.data_ptr(), 0, gen.STREAM_GRAD, step, nd, psi, 1e-2, 1.0,
                                  1, rank_stride=padded, cuda_stream=sp)
                z.zero_step(plan, grads, master, m, v, params, None, sp)
            gen.cuda_ranks_16(grads.data_ptr(), 0, gen.STREAM_GRAD, 6, nd, psi, 1e-2, 1.0, 1,
                              rank_stride=padded, cuda_stream=sp)
            small = (2 * nd + 14) * psi < (1 << 30)
            k = max(args.steps, 200 if small else 20)
            ms = _timed_steps(torch, stream,
                              lambda: z.zero_step(plan, grads, master, m, v, params, None, sp),
                              k, flush=flush if small else None) / k
            gbs = (2 * nd + 26) * psi / (ms / 1e3) / 1e9
            line.update({"ms_per_step": ms, "params_per_s": psi / (ms / 1e3),
                         "hbm_gbs_roofline_bytes": gbs, "roofline_bytes_per_elem": 2 * nd + 26,
                         "frac_of_measured_hbm": gbs / peak, "peak_gbs": peak, "steps": k,
                         "warmup": 5, "path": "fused single pass",
                         "l2": ("flushed between steps (256 MB written, then 256 MB read)"
                                if small else "inputs larger than L2")})
            print(json.dumps(line), flush=True)
            z.zero_plan_destroy(plan)
            del grads, master, m, v, params


def run_stage3(args):
    """LLaMA-3-8B at Nd = 64, ZeRO-3: one step = the update of rank 0's resident
    shard from its 64 contributions, then the gather of every unit (34) from the
    64 ranks' parameter shards into one buffer."""
    print(json.dumps(stage3_measure(args)), flush=True)


def stage3_measure(args) -> dict:
    """The measurements run_stage3 prints, as a dict (buffers freed on return)."""
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild
    zbuild.build()
    w = workload(name="llama3-8b")
    if args.layers or args.vocab:
        from gen import workloads as W
        w = W.scaled_llama(args.layers or 32, 4096, 14336, 32, 8, args.vocab or 128256, w.nd, w)
    if args.nd:
        w = dataclasses.replace(w, nd=args.nd)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    peak, _ = measured_peaks()
    plan = _plan_for(z, w, units=w.units)
    _, total, nunits, _ = z.zero_plan_layout(plan)
    units = [z.zero_plan_unit(plan, u) for u in range(nunits)]
    grads = torch.empty((w.nd, total), dtype=torch.int16, device=dev)
    master = torch.zeros(total, dtype=torch.float32, device=dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    params = torch.zeros(total, dtype=torch.int16, device=dev)
    shards = torch.empty((w.nd - 1, total), dtype=torch.int16, device=dev)
    out = torch.empty(max(u[0] for u in units), dtype=torch.int16, device=dev)
    gen.cuda_ranks_16(grads.data_ptr(), 0, gen.STREAM_GRAD, 1, w.nd, total, w.grad_sigma, 1.0,
                      w.dtype, cuda_stream=sp)
    gen.cuda_f32(master.data_ptr(), 0, gen.STREAM_MASTER, 0, 0, total, 0.02, cuda_stream=sp)
    for k in range(1, w.nd):
        gen.cuda_s16(shards[k - 1].data_ptr(), 0, gen.STREAM_SHARD, 0, k, total, 0.02, 1.0,
                     w.dtype, cuda_stream=sp)
    ptrs = [params.data_ptr()] + [shards[k].data_ptr() for k in range(w.nd - 1)]

    def update():
        z.zero_step(plan, grads, master, m, v, params, None, sp)

    def gather_all():
        for u in range(nunits):
            z.zero_gather_layer(plan, u, ptrs, out, sp)

    for _ in range(max(3, args.warmup)):
        update()
        gather_all()
    torch.cuda.synchronize()
    K = max(args.steps, 10)
    t_upd = _timed_steps(torch, stream, update, K) / K
    t_gat = _timed_steps(torch, stream, gather_all, K) / K
    upd_bytes = (2 * w.nd + 26) * total
    gat_bytes = 4 * w.psi
    qwz = {}
    if args.qwz:
        bits = args.qwz
        cbytes = total if bits == 8 else (total + 1) // 2
        codes = torch.empty((w.nd, cbytes + 16), dtype=torch.uint8, device=dev)
        scales = torch.empty((w.nd, -(-total // 256)), dtype=torch.float32, device=dev)
        z.zero_quantize_shard(w.dtype, params, total, bits, codes[0], scales[0], sp)
        for k in range(1, w.nd):
            z.zero_quantize_shard(w.dtype, shards[k - 1], total, bits, codes[k], scales[k], sp)
        cptr = [codes[k].data_ptr() for k in range(w.nd)]
        sptr = [scales[k].data_ptr() for k in range(w.nd)]

        def gather_all_q():
            z.zero_quantize_shard(w.dtype, params, total, bits, codes[0], scales[0], sp)
            for u in range(nunits):
                z.zero_gather_layer_q(plan, u, bits, cptr, sptr, out, sp)

        for _ in range(2):
            gather_all_q()
        t_q = _timed_steps(torch, stream, gather_all_q, K) / K
        q_bytes = (2 + bits / 8) * total + (bits / 8 + 2) * w.psi + 4 * w.psi / 256

        # the qwZ step as one update pass that quantizes in its epilogue, then
        # the quantized gathers
        def update_q():
            z.zero_step_qwz(plan, grads, master, m, v, params, None, bits, codes[0], scales[0],
                            sp)

        def gathers_q():
            for u in range(nunits):
                z.zero_gather_layer_q(plan, u, bits, cptr, sptr, out, sp)

        def step_q():
            update_q()
            gathers_q()

        for _ in range(2):
            step_q()
        t_uq = _timed_steps(torch, stream, update_q, K) / K
        t_gq = _timed_steps(torch, stream, gathers_q, K) / K
        t_sq = _timed_steps(torch, stream, step_q, K) / K
        uq_bytes = (2 * w.nd + 26 + bits / 8 + 4 / 256) * total
        gq_bytes = (bits / 8 + 2 + 4 / 256) * w.psi
        qwz = {"bits": bits, "block": 256, "quantize_and_gather_ms": t_q,
               "bytes_per_elem": bits / 8 + 2 + 4 / 256,
               "gbs": q_bytes / (t_q / 1e3) / 1e9,
               "vs_unquantized_gather": t_gat / t_q,
               "frac_of_measured_hbm": q_bytes / (t_q / 1e3) / 1e9 / peak,
               "fused_step": {
                   "what": "zero_step_qwz (update + quantize in one pass) then the quantized "
                           "gathers of every unit",
                   "step_ms": t_sq, "update_q_ms": t_uq, "gathers_q_ms": t_gq,
                   "update_q_gbs": uq_bytes / (t_uq / 1e3) / 1e9,
                   "update_q_frac_of_measured_hbm": uq_bytes / (t_uq / 1e3) / 1e9 / peak,
                   "gathers_q_frac_of_measured_hbm": gq_bytes / (t_gq / 1e3) / 1e9 / peak,
                   "vs_unquantized_step": (t_upd + t_gat) / t_sq,
                   "vs_separate_update_quantize_gather": (t_upd + t_q) / t_sq}}
    desc = DESCRIPTIONS.get(w.name, f"LLaMA-3-8B-shaped list scaled to {len(units) - 2} layers")
    res = {
        "mode": "zero3", "metric": "ZeRO-3 step: resident-shard update and per-unit gathers",
        "workload": f"{w.name}: {desc}, {len(w.shapes)} tensors, {nunits} units",
        "psi": w.psi, "nd": w.nd, "shard_elems": total, "steps": K,
        "update_ms": t_upd, "update_params_per_s": total / (t_upd / 1e3),
        "update_gbs": upd_bytes / (t_upd / 1e3) / 1e9, "update_bytes_per_elem": 2 * w.nd + 26,
        "gather_ms_all_units": t_gat, "gather_gbs": gat_bytes / (t_gat / 1e3) / 1e9,
        "gather_bytes_per_elem": 4, "step_ms": t_upd + t_gat,
        "frac_of_measured_hbm": {"update": upd_bytes / (t_upd / 1e3) / 1e9 / peak,
                                 "gather": gat_bytes / (t_gat / 1e3) / 1e9 / peak},
        "qwz": qwz or None,
        "l2": (f"inputs larger than L2 ({2 * w.nd * total / 1e9:.1f} GB gradients, "
               f"{2 * (w.nd - 1) * total / 1e9:.1f} GB shards)")}
    z.zero_plan_destroy(plan)
    return res


def run_buckets(args):
    """Bucketed steps on the named workload: constant-size gradient buckets
    (two buffers of nd x B 16-bit values) instead of the full nd x padded
    gradients.  Times the bucket reduces + update alone, the synthetic backward
    producer alone (the input generator filling each bucket, last bucket first),
    and the two overlapped on two streams."""
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild
    zbuild.build()
    w = workload(args.psi, args.workload, args.nd)
    dev = torch.device("cuda", 0)
    peak, _ = measured_peaks()
    plan = _plan_for(z, w)
    B = args.buckets
    ws = z.zero_plan_set_bucket(plan, B)
    _, padded, _, _ = z.zero_plan_layout(plan)
    n = w.psi
    nb = -(-n // B)
    master = torch.zeros(padded, dtype=torch.float32, device=dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    params = torch.zeros(padded, dtype=torch.int16, device=dev)
    work = torch.empty(ws // 4, dtype=torch.float32, device=dev)
    bufs = [torch.empty((w.nd, B), dtype=torch.int16, device=dev) for _ in range(2)]
    producer, consumer = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    gen.cuda_f32(master.data_ptr(), 0, gen.STREAM_MASTER, 0, 0, n, 0.02,
                 cuda_stream=consumer.cuda_stream)

    def produce(j, b, step):
        first, count = b * B, min(B, n - b * B)
        gen.cuda_ranks_16(bufs[j % 2].data_ptr(), 0, gen.STREAM_GRAD, step, w.nd, count,
                          w.grad_sigma, w.loss_scale, w.dtype, rank_stride=B, index0=first,
                          cuda_stream=producer.cuda_stream)

    order = list(range(nb))[::-1]

    def pipelined(step):
        freed = [None, None]
        for j, b in enumerate(order):
            if freed[j % 2] is not None:
                producer.wait_event(freed[j % 2])
            produce(j, b, step)
            ready = torch.cuda.Event()
            ready.record(producer)
            consumer.wait_event(ready)
            z.zero_step_bucket(plan, b, bufs[j % 2], work, consumer.cuda_stream)
            done = torch.cuda.Event()
            done.record(consumer)
            freed[j % 2] = done
        z.zero_step_apply(plan, master, m, v, params, work, consumer.cuda_stream)

    def reduce_only():
        for j, b in enumerate(order):
            z.zero_step_bucket(plan, b, bufs[j % 2], work, consumer.cuda_stream)
        z.zero_step_apply(plan, master, m, v, params, work, consumer.cuda_stream)

    def produce_only(step):
        for j, b in enumerate(order):
            produce(j, b, step)

    def timed(fn, stream, k):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(k):
            fn(i)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / k * 1e3

    for i in range(max(3, args.warmup)):
        pipelined(i + 1)
    K = max(5, min(args.steps, 20))
    t_pipe = timed(lambda i: pipelined(i + 1), consumer, K)
    t_red = timed(lambda i: reduce_only(), consumer, K)
    t_prod = timed(lambda i: produce_only(i + 1), producer, K)
    step_bytes = (2 * w.nd + 26) * n
    print(json.dumps({
        "mode": "buckets", "metric": "bucketed step: constant-size gradient buckets",
        "workload": f"{w.name}: {DESCRIPTIONS.get(w.name, w.name)}", "psi": n, "nd": w.nd,
        "bucket_elems": B, "buckets": nb,
        "gradient_staging_bytes": 2 * w.nd * B * 2, "full_gradient_bytes": w.nd * padded * 2,
        "reduce_and_apply_ms": t_red, "producer_ms": t_prod, "pipelined_ms": t_pipe,
        "overlap": (t_red + t_prod) / t_pipe,
        "hbm_gbs_roofline_bytes_reduce_and_apply": step_bytes / (t_red / 1e3) / 1e9,
        "frac_of_measured_hbm": step_bytes / (t_red / 1e3) / 1e9 / peak,
        "timing": "host wall clock around K steps with device synchronisation"}), flush=True)
    z.zero_plan_destroy(plan)


def run_checkpoint(args):
    """Sharded checkpoint of the workload's optimizer state through the C ABI:
    every rank's file saved (into the page cache, then flushed to storage with
    the files' cached pages dropped), then loaded into a plan at half the rank
    count (a reshard) from storage and again from the page cache.  Wall-clock
    times of the synchronous calls; loaded state checked on sampled elements."""
    import dataclasses
    import shutil
    import tempfile
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild
    zbuild.build()
    w = workload(args.psi, args.workload, args.nd)
    if w.stage == 3:
        print(json.dumps({"mode": "checkpoint", "workload": w.name,
                          "unavailable": "a ZeRO-3 plan holds one rank's shard; this mode "
                                         "saves every rank of a stages 0-2 plan"}), flush=True)
        return
    dev = torch.device("cuda", 0)
    state_bytes = 14 * w.psi                      # master, m, v (fp32) + 16-bit params
    base = args.ckpt_dir or tempfile.gettempdir()
    free = shutil.disk_usage(base).free
    line = {"mode": "checkpoint", "workload": f"{w.name}: {DESCRIPTIONS.get(w.name, w.name)}",
            "psi": w.psi, "nd_saved": w.nd, "nd_loaded": max(1, w.nd // 2),
            "checkpoint_bytes": state_bytes, "dir_free_bytes": free}
    if free < 2.5 * state_bytes:
        line["unavailable"] = f"{base} has {free} bytes free; needs {int(2.5 * state_bytes)}"
        print(json.dumps(line), flush=True)
        return
    d = tempfile.mkdtemp(prefix="zck_", dir=base)
    plan = _plan_for(z, w)
    w2 = dataclasses.replace(w, nd=max(1, w.nd // 2))
    plan2 = _plan_for(z, w2)
    try:
        _, padded, _, _ = z.zero_plan_layout(plan)
        _, padded2, _, _ = z.zero_plan_layout(plan2)
        a = [torch.zeros(padded, dtype=torch.float32, device=dev) for _ in range(3)]
        a.append(torch.zeros(padded, dtype=torch.int16, device=dev))
        gen.cuda_f32(a[0].data_ptr(), 0, gen.STREAM_MASTER, 0, 0, w.psi, 0.02)
        a[1][:w.psi].normal_()
        a[2][:w.psi].uniform_()
        a[3][:w.psi].random_(-32768, 32767)
        b = [torch.full((padded2,), 3.0, dtype=torch.float32, device=dev) for _ in range(3)]
        b.append(torch.full((padded2,), 7, dtype=torch.int16, device=dev))
        torch.cuda.synchronize()

        def clock(fn):
            t0 = time.perf_counter()
            fn()
            return time.perf_counter() - t0

        t = {}
        flags = z.ZERO_CKPT_FSYNC | z.ZERO_CKPT_DROP_CACHE
        t["save_fsync"] = clock(lambda: z.zero_checkpoint_save(plan, d + "/s", -1, *a, flags))
        t["load_after_drop"] = clock(lambda: z.zero_checkpoint_load(plan2, d + "/s", -1, *b))
        t["load_page_cache"] = clock(lambda: z.zero_checkpoint_load(plan2, d + "/s", -1, *b))
        idx = torch.randint(0, w.psi, (1 << 20,), device=dev)
        ok = all(torch.equal(x[idx], y[idx]) for x, y in zip(a, b))
        ok = ok and not any(bool(y[w.psi:].any()) for y in b)
        os.sync()
        t["save_page_cache"] = clock(lambda: z.zero_checkpoint_save(plan, d + "/c", -1, *a))
        shutil.rmtree(d + "/c")
        os.sync()
        # the device<->host link, for scale: one pinned copy each way
        nl = min(1 << 28, padded)
        host = torch.empty(nl, dtype=torch.float32, pin_memory=True)
        src = a[0][:nl]
        for _ in range(2):
            host.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        host.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        d2h = nl * 4 / (time.perf_counter() - t0) / 1e9
        t0 = time.perf_counter()
        src.copy_(host, non_blocking=True)
        torch.cuda.synchronize()
        h2d = nl * 4 / (time.perf_counter() - t0) / 1e9
        # the storage under `base`, for scale: dd of 4 GiB, flushed / read direct
        dd = {}
        ddf = d + "/dd.bin"
        try:
            t0 = time.perf_counter()
            subprocess.run(["dd", "if=/dev/zero", f"of={ddf}", "bs=64M", "count=64",
                            "conv=fsync"], check=True, capture_output=True)
            dd["dd_write_fsync_gbs"] = (64 << 26) / (time.perf_counter() - t0) / 1e9
            t0 = time.perf_counter()
            subprocess.run(["dd", f"if={ddf}", "of=/dev/null", "bs=64M", "iflag=direct"],
                           check=True, capture_output=True)
            dd["dd_read_direct_gbs"] = (64 << 26) / (time.perf_counter() - t0) / 1e9
        except (OSError, subprocess.CalledProcessError) as e:
            dd["dd"] = f"not measured: {e}"
        line.update({f"{k}_s": v for k, v in t.items()})
        line.update({f"{k}_gbs": state_bytes / v / 1e9 for k, v in t.items()})
        line.update(dd)
        line.update({"link_d2h_gbs": d2h, "link_h2d_gbs": h2d, "verified_sample": bool(ok),
                     "host_threads": os.cpu_count(), "dir": base,
                     "timing": "host wall clock around each synchronous call"})
        print(json.dumps(line), flush=True)
    finally:
        z.zero_plan_destroy(plan)
        z.zero_plan_destroy(plan2)
        shutil.rmtree(d, ignore_errors=True)


def host_copy_gbs(threads, nbytes=4 << 30):
    """Host memory bandwidth for scale: `threads` threads each copying their slice
    of an nbytes array (numpy copies release the GIL); read + write bytes / s.
    The arrays sit on transparent huge pages, like the offload leg's host state."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    src = huge_host_array(nbytes // 4, np.float32)
    src[:] = 1.0
    dst = huge_host_array(nbytes // 4, np.float32)
    parts = np.array_split(np.arange(src.size), threads)
    bounds = [(int(p[0]), int(p[-1]) + 1) for p in parts if p.size]

    def one(b):
        np.copyto(dst[b[0]:b[1]], src[b[0]:b[1]])

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(one, bounds))                   # first touch
        best = 0.0
        for _ in range(3):
            t0 = time.perf_counter()
            list(ex.map(one, bounds))
            best = max(best, 2 * nbytes / (time.perf_counter() - t0) / 1e9)
    return best


def run_offload(args):
    """ZeRO-Offload on the workload: the device reduce (16-bit averaged gradient),
    the copy to the host, the host Adam on host-resident master, m, v and the
    16-bit parameters back, through zero_offload_step; and the host Adam alone
    (zero_cpu_adam).  Wall clock around the synchronous calls."""
    import numpy as np
    import torch
    import gen
    import zero_sharded_mixed_02_gb300 as z
    from zero_sharded_mixed_02_gb300 import build as zbuild
    zbuild.build()
    w = workload(args.psi, args.workload, args.nd)
    if w.stage == 3:
        print(json.dumps({"mode": "offload", "workload": w.name,
                          "unavailable": "offload runs on stages 0-2 plans"}), flush=True)
        return
    dev = torch.device("cuda", 0)
    plan = _plan_for(z, w)
    threads = args.host_threads or os.cpu_count()
    try:
        _, padded, _, _ = z.zero_plan_layout(plan)
        n = w.psi
        d = torch.zeros(padded, dtype=torch.float32, device=dev)
        gen.cuda_f32(d.data_ptr(), 0, gen.STREAM_MASTER, 0, 0, n, 0.02)
        # host state on transparent huge pages (the host Adam streams 28 bytes
        # per parameter through these arrays every step)
        master = huge_host_array(padded, np.float32)
        master[:] = d.cpu().numpy()
        del d
        m = huge_host_array(padded, np.float32)
        v = huge_host_array(padded, np.float32)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(padded, dtype=torch.int16, device=dev)
        grads = torch.empty((w.nd, padded), dtype=torch.int16, device=dev)
        gen.cuda_ranks_16(grads.data_ptr(), 0, gen.STREAM_GRAD, 1, w.nd, n, w.grad_sigma,
                          w.loss_scale, w.dtype, rank_stride=padded)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream().cuda_stream
        for _ in range(max(1, args.warmup)):
            z.zero_offload_step(plan, grads, master, m, v, params, work, threads, stream)
        K = max(2, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(K):
            z.zero_offload_step(plan, grads, master, m, v, params, work, threads, stream)
        t_step = (time.perf_counter() - t0) / K
        r = z.zero_step_result(plan)
        # the host Adam alone, on the last copied gradient
        g16 = huge_host_array(n, np.uint16)
        g16[:] = work[:n].cpu().numpy()
        p16 = huge_host_array(n, np.uint16)
        hp = z.hparams(**w.hparams())
        z.zero_cpu_adam(g16, w.dtype, n, r["loss_scale"], 1.0, 0.5, 0.5, hp, master, m, v,
                        p16, threads)
        t0 = time.perf_counter()
        for _ in range(K):
            z.zero_cpu_adam(g16, w.dtype, n, r["loss_scale"], 1.0, 0.5, 0.5, hp, master, m, v,
                            p16, threads)
        t_adam = (time.perf_counter() - t0) / K
        bw = host_copy_gbs(threads)
        host_bytes = 28 * n          # g16 2 + master/m/v 12 read, 12 written, params 2 written
        print(json.dumps({
            "mode": "offload", "workload": f"{w.name}: {DESCRIPTIONS.get(w.name, w.name)}",
            "psi": n, "nd": w.nd, "host_threads": threads,
            "offload_step_ms": t_step * 1e3, "offload_step_params_per_s": n / t_step,
            "host_adam_ms": t_adam * 1e3, "host_adam_params_per_s": n / t_adam,
            "pages_cpu_adam_params_per_s": 1.5e9,
            "host_adam_vs_pages": n / t_adam / 1.5e9,
            "host_adam_gbs": host_bytes / t_adam / 1e9, "host_copy_gbs_measured": bw,
            "host_adam_frac_of_copy": host_bytes / t_adam / 1e9 / bw,
            "link_bytes_per_step": 4 * n, "step_result": r,
            "timing": "host wall clock around the synchronous calls"}), flush=True)
    finally:
        z.zero_plan_destroy(plan)


# ------------------------------------------------------------ reference arm
def run_reference(args):
    """The CPU oracle, as it stands, on the host cores: each step is one oracle
    step over a bounded sample of the same workload."""
    rank, _, ws = dist_env()
    if rank != 0:
        return
    w = workload(args.psi, args.workload, args.nd)
    thr = oracle_threads(w.nd)
    n_s = args.ref_sample
    import oracle
    padded = oracle.shard_elems(w.psi, w.nd) * w.nd
    oracle_sample(w, n_s, thr, max_repeats=max(1, args.warmup))          # warm-up
    pps, per, reps = oracle_sample(w, n_s, thr, max_repeats=args.steps)
    out = {
        "impl": "reference", "metric": metric_of(w), "value": pps, "unit": "params/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded counter-based generator; shape list only, no weights)",
        "config": config_of(w, padded),
        "cpu_baseline": {"value": pps, "unit": "params/s", "cores": thr, "kind": "oracle",
                         "sample": f"first {n_s} elements x {w.nd} ranks per step"},
        "e2e": {"value": pps, "unit": "params/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the other workloads measured after the headline")
    ap.add_argument("--cpu-sample", type=int, default=1 << 23)
    ap.add_argument("--ref-sample", type=int, default=1 << 21)
    ap.add_argument("--reduce-kernel", choices=("ldg", "tma"), default="ldg",
                    help="reduce-pass kernel: 128-bit loads (default) or TMA bulk staging")
    ap.add_argument("--workload", choices=WORKLOADS, default="gpt2-1.5b")
    ap.add_argument("--sweep", action="store_true",
                    help="bandwidth sweep: one JSON line per (psi, nd) point")
    ap.add_argument("--pingpong", action="store_true",
                    help="the workload with its clip off: zero_step against zero_step_pingpong")
    ap.add_argument("--offload", action="store_true",
                    help="time ZeRO-Offload steps (device reduce, host Adam) on the workload")
    ap.add_argument("--host-threads", type=int, default=0, help="host threads for --offload")
    ap.add_argument("--checkpoint", action="store_true",
                    help="time a sharded checkpoint save and a resharding load of the workload")
    ap.add_argument("--ckpt-dir", default=None, help="where --checkpoint writes (default: tmp)")
    ap.add_argument("--buckets", type=int, default=0,
                    help="bucketed steps with buckets of this many elements (a multiple of 64)")
    ap.add_argument("--qwz", type=int, choices=(0, 4, 8), default=0,
                    help="ZeRO-3 workload: also time the quantized (qwZ) gather at this width")
    ap.add_argument("--psi", type=int, default=0,
                    help="flat model of this many parameters (profiling small cases); "
                         "with --sweep, this one psi")
    ap.add_argument("--nd", type=int, default=0,
                    help="ranks of the --psi flat model or the llama3-8b workload; "
                         "with --sweep, this one nd")
    ap.add_argument("--layers", type=int, default=0,
                    help="llama3-8b workload: this many transformer layers (small cases)")
    ap.add_argument("--vocab", type=int, default=0,
                    help="llama3-8b workload: this vocabulary size (small cases)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.buckets:
        run_buckets(args)
    elif args.checkpoint:
        run_checkpoint(args)
    elif args.offload:
        run_offload(args)
    elif args.pingpong:
        run_pingpong(args)
    elif args.workload == "llama3-8b":
        run_stage3(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
