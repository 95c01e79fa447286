"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on the
same seeded inputs, at sizes the oracle finishes in seconds that still span many
blocks and a ragged tail.  Tolerances are in tests/harness.py."""
import dataclasses

import numpy as np
import pytest

import gen
import harness as H
import oracle
from gen import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def z():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_sharded_mixed_02_gb300 import build
    build.build()
    import zero_sharded_mixed_02_gb300 as z
    z.lib()
    return z


def check(z, c, g32=False, reduce_kernel=0):
    """The case through the library and through the oracle (which admits the
    GPU's clip coefficient when it is within the harness's bound of its own);
    results by the harness's rules and the state bit for bit."""
    gpu = H.run_gpu(z, c, keep_g32=g32, reduce_kernel=reduce_kernel)
    n = gpu.master.size
    padded = n
    if c.stage <= 2:
        plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z))
        padded = z.zero_plan_layout(plan)[1]
        z.zero_plan_destroy(plan)
        mask = None
    else:
        plan = z.zero_plan_create(c.psi, c.nd, 3, c.dtype, c.shapes, c.hparams(z), units=c.units)
        mask = H.stage3_valid_mask(z, plan, c.nd)
        z.zero_plan_destroy(plan)
    ora = H.run_oracle(c, n, padded, mask, follow=gpu.results)
    H.compare_runs(gpu, ora, what=f"psi={c.psi} nd={c.nd}")
    H.assert_state_equal(gpu, ora, what=f"psi={c.psi} nd={c.nd}")
    if g32:
        # the reduced (averaged, unscaled) gradient of the last step is bit-exact
        last = c.steps
        scale = gpu.results[-2]["loss_scale"] if c.steps > 1 else c.loss_scale
        g = H.grads_for_step(c, last, n, padded, scale, mask)
        want, _ = oracle.reduce(c.nd, c.dtype, np.ascontiguousarray(g[:, :n]), loss_scale=scale)
        assert np.array_equal(gpu.g32.view(np.uint32), want.view(np.uint32))
    return gpu, ora


def test_tiny_flat_model(z):
    # tiny flat model: 4 tensors, Nd=4, ZeRO-2, fp16 x1024 dynamic loss scale, 3 steps
    c = H.from_workload(W.tiny())
    gpu, ora = check(z, c, g32=True)
    assert [r["t"] for r in gpu.results] == [1, 2, 3]


def test_gpt2_small_family(z):
    # GPT-2 small's settings (Nd=8, ZeRO-1, bf16, AdamW 0.01, clip 1.0, 10 steps)
    # on a 2-layer model of the same shape family
    w = W.scaled_gpt2(2, 256, 1024, 1000, 128, 8, W.gpt2_small())
    c = H.from_workload(w)
    gpu, _ = check(z, c, g32=True)
    assert all(r["clip_coef"] < 1.0 for r in gpu.results)      # the clip is active


def test_gpt2_xl_family_with_overflow(z):
    # GPT-2 1.5B's settings (Nd=16, ZeRO-2, fp16 x65536 dynamic, clip 1, inf on
    # steps 3 and 7: skipped, scale halved) on a 2-layer model of the same family
    w = W.scaled_gpt2(2, 320, 1280, 3000, 256, 16, W.gpt2_xl())
    c = H.from_workload(w)
    gpu, _ = check(z, c, g32=True)
    skipped = [r["skipped"] for r in gpu.results]
    assert skipped == [0, 0, 1, 0, 0, 0, 1, 0, 0, 0]
    assert gpu.results[-1]["loss_scale"] == 16384.0 and gpu.results[-1]["t"] == 8


def test_llama_family_stage3_and_gather(z):
    # LLaMA-3-8B's settings (Nd=64, ZeRO-3, bf16): rank 0's shard updated, then
    # every unit gathered from 64 shards (rank 0's updated one + 63 seeded)
    import torch
    w = W.scaled_llama(2, 256, 512, 8, 2, 1000, 64, W.llama3_8b())
    c = H.from_workload(w, steps=2)
    plans = []
    gpu = H.run_gpu(z, c, plan_out=plans)
    plan = plans[0]
    try:
        _, total, nunits, _ = z.zero_plan_layout(plan)
        assert nunits == 4
        mask = H.stage3_valid_mask(z, plan, c.nd)
        ora = H.run_oracle(c, total, total, mask, follow=gpu.results)
        H.compare_runs(gpu, ora, "stage3")
        H.assert_state_equal(gpu, ora, "stage3")
        dev = torch.device("cuda", 0)
        shards = [torch.from_numpy(gpu.params.view(np.int16)).to(dev)]
        host_shards = [gpu.params]
        for k in range(1, c.nd):
            s = gen.s16(c.seed, gen.STREAM_SHARD, 0, k, total, 0.02, 1.0, c.dtype)
            s[~H.stage3_valid_mask(z, plan, c.nd, rank=k)] = 0
            host_shards.append(s)
            shards.append(torch.from_numpy(s.view(np.int16)).to(dev))
        for u in range(nunits):
            ln, sl, off = z.zero_plan_unit(plan, u)
            out = torch.full((ln + 8,), -1, dtype=torch.int16, device=dev)
            z.zero_gather_layer(plan, u, shards, out, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            got = out.cpu().numpy().view(np.uint16)
            want = oracle.gather_unit(c.nd, ln, sl, [s[off:off + sl] for s in host_shards])
            assert np.array_equal(got[:ln], want)
            assert np.all(got[ln:] == 0xFFFF)                     # nothing past the unit
    finally:
        z.zero_plan_destroy(plan)


@pytest.mark.parametrize("nd", [1, 2, 8, 32])
def test_bandwidth_sweep_point(z, nd):
    # the sweep's flat bf16 model (no clip, no loss scale: the fused single pass),
    # 5 warm-up steps + 1; every output bit-exact
    c = H.Case(shapes=[(1 << 20,)], nd=nd, steps=6)
    check(z, c)


EDGE = []
for psi in (1, 5, 13, 16, 4099, 65539):
    for nd in (1, 2, 3, 5, 8, 16):
        EDGE.append((psi, nd))


@pytest.mark.parametrize("psi,nd", EDGE)
@pytest.mark.parametrize("mode", ["fused", "clip", "fp16-dyn"])
def test_edge_sizes(z, psi, nd, mode):
    shapes = [(psi,)] if psi < 100 else [(psi - 7,), (7,)]
    if mode == "fused":
        c = H.Case(shapes=shapes, nd=nd, steps=3, weight_decay=0.01, decoupled_wd=0)
    elif mode == "clip":
        c = H.Case(shapes=shapes, nd=nd, steps=3, clip=0.05, weight_decay=0.01)
    else:
        c = H.Case(shapes=shapes, nd=nd, steps=4, dtype=gen.FP16, grad_sigma=1e-3,
                   loss_scale=4096.0, dynamic_scale=1, inf_steps=(2,), growth_interval=2)
    check(z, c, g32=(mode != "fused" and nd >= 4))


def test_nan_and_inf_skip_and_scale_schedule(z):
    c = H.Case(shapes=[(3000,), (1000,)], nd=4, dtype=gen.FP16, grad_sigma=1e-3,
               loss_scale=1024.0, dynamic_scale=1, steps=7, inf_steps=(2,), nan_steps=(5,),
               growth_interval=2)
    gpu, _ = check(z, c)
    assert [r["skipped"] for r in gpu.results] == [0, 1, 0, 0, 1, 0, 0]
    assert [r["loss_scale"] for r in gpu.results] == [1024, 512, 512, 1024, 512, 512, 1024]


STATIC_OVERFLOW = {
    # name: (case settings, kernel path the plan must take)
    "fused-no-clip": (dict(nd=8, dtype=gen.BF16), 0),
    "two-pass-clip": (dict(nd=8, dtype=gen.BF16, clip=1.0), 1),
    "recompute-clip": (dict(nd=2, dtype=gen.BF16, clip=1.0), 2),
    "fp16-scaled-clip": (dict(nd=4, dtype=gen.FP16, grad_sigma=1e-3, loss_scale=8.0, clip=1.0),
                         1),
    "skip-on-overflow": (dict(nd=4, dtype=gen.FP16, grad_sigma=1e-3, loss_scale=8.0,
                              skip_on_overflow=1), 1),
    "skip-on-overflow-recompute": (dict(nd=3, dtype=gen.BF16, skip_on_overflow=1, clip=1.0), 2),
}


@pytest.mark.parametrize("name", sorted(STATIC_OVERFLOW))
def test_static_scale_overflow_against_the_oracle(z, name):
    """Overflow under a static loss scale, against the oracle's state and
    results over the steps that follow: without skip_on_overflow the flag is
    reported and the step goes ahead (no clip: only the planted element turns
    non-finite; clip: tau / inf = 0 makes every other element take a
    zero-gradient step); with it the step is skipped and the scale kept.  +inf
    at step 2, NaN at step 4, 5 steps; every other element bit-exact."""
    over, path = STATIC_OVERFLOW[name]
    c = H.Case(shapes=[(40_000,), (1_003,)], steps=5, inf_steps=(2,), nan_steps=(4,), **over)
    plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z))
    assert z.zero_plan_path(plan) == path
    z.zero_plan_destroy(plan)
    gpu, ora = check(z, c)
    assert [r["overflow"] for r in gpu.results] == [0, 1, 0, 1, 0]
    skip = c.skip_on_overflow
    assert [r["skipped"] for r in gpu.results] == [0, skip, 0, skip, 0]
    assert gpu.results[-1]["t"] == (3 if skip else 5)
    assert all(r["loss_scale"] == c.loss_scale for r in gpu.results)
    bad = np.isnan(ora.master)
    assert bad.any() == (not skip) and np.array_equal(bad, np.isnan(gpu.master))
    if not skip and not c.clip:
        assert bad.sum() == 2                      # the two planted elements only


NORM_RANGE = {
    # name: case settings.  The per-group binary32 sum of squares q of 8 averaged
    # gradients goes to the thread's binary32 pair when 2^-60 <= q <= 2^100 and to
    # its binary64 part otherwise; sigma puts the groups across a boundary (both
    # parts in use in every block) or wholly past it.
    "edge-high": dict(grad_sigma=8.3e14, clip=1.0),
    "edge-low": dict(grad_sigma=6.9e-10, clip=1e-8),
    "past-high": dict(grad_sigma=1e20, clip=1.0),
    "past-low": dict(grad_sigma=1e-25, clip=1e-30),
    "edge-low-no-clip": dict(grad_sigma=6.9e-10),
}


@pytest.mark.parametrize("name", sorted(NORM_RANGE))
def test_norm_across_binary32_range(z, name):
    """bf16 gradients whose squares leave binary32's comfortable range: the norm
    against the oracle's binary64 sum (within the harness's bound; the clip
    coefficient it gives admitted within 8 ulp), and the state bit for bit."""
    c = H.Case(shapes=[(40_000,), (1_003,)], nd=4, steps=3, dtype=gen.BF16, **NORM_RANGE[name])
    gpu, ora = check(z, c)
    assert all(np.isfinite(r["grad_norm"]) and r["grad_norm"] > 0 for r in gpu.results)
    if c.clip:
        assert all(r["clip_coef"] < 1.0 for r in gpu.results)


HOST_GRADS = {
    # name: (case settings, kernel path)
    "two-pass-clip": (dict(shapes=[(300_001,), (77,)], nd=16, dtype=gen.FP16, grad_sigma=1e-3,
                           loss_scale=4096.0, dynamic_scale=1, clip=0.5, inf_steps=(2,)), 1),
    "fused": (dict(shapes=[(200_003,)], nd=8), 0),
    "recompute": (dict(shapes=[(200_003,)], nd=2, clip=1.0), 2),
    "stage3": (dict(shapes=[(5000,), (77,), (3000, 3)], units=[0, 0, 1], nd=8, stage=3,
                    clip=1.0), 1),
}


@pytest.mark.parametrize("name", sorted(HOST_GRADS))
def test_grads_in_page_locked_host_memory(z, name):
    """zero_step given the ranks' gradients in page-locked host memory (read in
    place over the host link) leaves the state and reports the results of the
    same steps from device memory, bit for bit."""
    over, path = HOST_GRADS[name]
    c = H.Case(steps=4, **over)
    plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z),
                              units=c.units if c.stage == 3 else None)
    assert z.zero_plan_path(plan) == path
    z.zero_plan_destroy(plan)
    a = H.run_gpu(z, c)
    b = H.run_gpu(z, c, grads_on_host=True)
    assert a.results == b.results
    for x, y in zip((a.master, a.m, a.v, a.params), (b.master, b.m, b.v, b.params)):
        assert x.tobytes() == y.tobytes()


def test_empty_model(z):
    plan = z.zero_plan_create(0, 4, 2, 1, [], z.hparams())
    try:
        for _ in range(3):
            z.zero_step(plan, None, None, None, None, None, None, 0)
        r = z.zero_step_result(plan)
        assert r["t"] == 3 and r["grad_norm"] == 0.0 and r["skipped"] == 0
    finally:
        z.zero_plan_destroy(plan)


def test_deterministic_rerun(z):
    c = H.Case(shapes=[(300_001,)], nd=8, clip=0.5, steps=3)
    a = H.run_gpu(z, c)
    b = H.run_gpu(z, c)
    for x, y in zip((a.master, a.m, a.v, a.params), (b.master, b.m, b.v, b.params)):
        assert x.tobytes() == y.tobytes()
    assert [r["grad_norm"] for r in a.results] == [r["grad_norm"] for r in b.results]


@pytest.mark.parametrize("nd", [3, 8])
def test_stages_0_1_2_are_bitwise_identical(z, nd):
    """Plain DP, ZeRO-1 and ZeRO-2 differ only in what each rank keeps in memory
    ([L18] 2.1-2.3): the step's results are the same bits."""
    c = H.Case(shapes=[(300_001,), (77,)], nd=nd, dtype=gen.FP16, grad_sigma=1e-3,
               loss_scale=4096.0, dynamic_scale=1, clip=0.5, steps=3, inf_steps=(2,))
    runs = [H.run_gpu(z, dataclasses.replace(c, stage=s)) for s in (0, 1, 2)]
    for r in runs[1:]:
        for x, y in zip((runs[0].master, runs[0].m, runs[0].v, runs[0].params),
                        (r.master, r.m, r.v, r.params)):
            assert x.tobytes() == y.tobytes()
        assert r.results == runs[0].results


def test_misaligned_and_missing_pointers_rejected(z):
    import torch
    c = H.Case(shapes=[(4096,)], nd=4, clip=1.0)
    plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        _, padded, _, ws = z.zero_plan_layout(plan)
        dev = torch.device("cuda", 0)
        g = torch.zeros((4, padded), dtype=torch.int16, device=dev)
        f = [torch.zeros(padded + 4, dtype=torch.float32, device=dev) for _ in range(3)]
        p = torch.zeros(padded, dtype=torch.int16, device=dev)
        w = torch.zeros(ws // 4, dtype=torch.float32, device=dev)
        with pytest.raises(z.ZeroError):
            z.zero_step(plan, g.data_ptr() + 2, f[0], f[1], f[2], p, w)
        with pytest.raises(z.ZeroError):
            z.zero_step(plan, g, f[0].data_ptr() + 4, f[1], f[2], p, w)
        with pytest.raises(z.ZeroError):
            z.zero_step(plan, g, f[0], f[1], f[2], p, None)         # workspace needed
        z.zero_step(plan, g, f[0], f[1], f[2], p, w)
        assert z.zero_step_result(plan)["t"] == 1
    finally:
        z.zero_plan_destroy(plan)


def test_profile_counts_kernels(z):
    import torch
    c = H.Case(shapes=[(100_000,)], nd=8, clip=1.0, steps=1)
    plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        _, padded, _, ws = z.zero_plan_layout(plan)
        dev = torch.device("cuda", 0)
        g = torch.zeros((8, padded), dtype=torch.int16, device=dev)
        f = [torch.zeros(padded, dtype=torch.float32, device=dev) for _ in range(3)]
        p = torch.zeros(padded, dtype=torch.int16, device=dev)
        w = torch.zeros(ws // 4, dtype=torch.float32, device=dev)
        z.zero_plan_profile(plan, 1)
        for _ in range(300):                                  # more than the event ring
            z.zero_step(plan, g, f[0], f[1], f[2], p, w)
        t = z.zero_plan_kernel_times(plan)
        assert t["steps"] == 300 and t["launches"] == 600
        assert t["reduce_ms"] > 0 and t["update_ms"] > 0
        assert z.zero_plan_path(plan) == z.PATH_G32
    finally:
        z.zero_plan_destroy(plan)


@pytest.mark.parametrize("psi,nd,dtype", [(1_000_003, 16, gen.FP16), (4096 * 7, 5, gen.BF16),
                                          (1000, 4, gen.FP16), (300_000, 32, gen.BF16),
                                          (1 << 20, 8, gen.FP16), (2048 + 8, 48, gen.BF16)])
def test_tma_staged_reduce(z, psi, nd, dtype):
    # the reduce pass with TMA bulk staging of the rank rows: same reduced gradient
    # bit for bit, same flags and skips; sizes below, at and off the 1024-element tile
    if dtype == gen.FP16:
        c = H.Case(shapes=[(psi,)], nd=nd, dtype=dtype, grad_sigma=1e-3, loss_scale=2048.0,
                   dynamic_scale=1, clip=1.0, steps=4, inf_steps=(2,))
    else:
        c = H.Case(shapes=[(psi,)], nd=nd, clip=0.5, steps=3, weight_decay=0.01)
    check(z, c, g32=True, reduce_kernel=1)


def test_tma_staged_reduce_skip_on_overflow(z):
    # static bf16 scale with skip_on_overflow through the TMA-staged reduce: the
    # step with +inf is skipped, the scale kept, the reduced gradient bit-exact
    c = H.Case(shapes=[(300_000,)], nd=16, skip_on_overflow=1, steps=3, inf_steps=(2,))
    gpu, _ = check(z, c, g32=True, reduce_kernel=1)
    assert [r["skipped"] for r in gpu.results] == [0, 1, 0]


def test_tma_staged_reduce_rejects_unsupported(z):
    for nd, kw in ((2, dict(clip=1.0)), (8, dict()), (64, dict(clip=1.0))):
        c = H.Case(shapes=[(4096,)], nd=nd, **kw)
        plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
        try:
            with pytest.raises(z.ZeroError):
                z.zero_plan_set_reduce_kernel(plan, 1)
            z.zero_plan_set_reduce_kernel(plan, 0)
        finally:
            z.zero_plan_destroy(plan)


def test_profile_fused_path_has_no_update_pass(z):
    import torch
    c = H.Case(shapes=[(100_000,)], nd=4, steps=1)              # no clip, no dynamic scale
    plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        assert z.zero_plan_path(plan) == z.PATH_FUSED
        _, padded, _, _ = z.zero_plan_layout(plan)
        dev = torch.device("cuda", 0)
        g = torch.zeros((4, padded), dtype=torch.int16, device=dev)
        f = [torch.zeros(padded, dtype=torch.float32, device=dev) for _ in range(3)]
        p = torch.zeros(padded, dtype=torch.int16, device=dev)
        z.zero_plan_profile(plan, 1)
        for _ in range(10):
            z.zero_step(plan, g, f[0], f[1], f[2], p, None)
        t = z.zero_plan_kernel_times(plan)
        assert t["steps"] == 10 and t["launches"] == 10
        assert t["reduce_ms"] > 0 and t["update_ms"] == 0.0
    finally:
        z.zero_plan_destroy(plan)


# ---- the largest rank counts the boundary accepts (nd up to 1024) ----
@pytest.mark.parametrize("nd", [1000, 1024])
@pytest.mark.parametrize("mode", ["clip", "fp16-dyn"])
def test_largest_rank_counts(z, nd, mode):
    # the generic-nd fold over up to 1024 rank rows; shards of 128 elements
    shapes = [(70_001,), (13,)]
    if mode == "clip":
        c = H.Case(shapes=shapes, nd=nd, steps=2, clip=0.05, weight_decay=0.01)
    else:
        c = H.Case(shapes=shapes, nd=nd, steps=3, dtype=gen.FP16, grad_sigma=1e-3,
                   loss_scale=4096.0, dynamic_scale=1, inf_steps=(2,))
    gpu, _ = check(z, c, g32=True)
    if mode != "clip":
        assert [r["skipped"] for r in gpu.results] == [0, 1, 0]


def test_largest_rank_count_stage3_gathers(z):
    # ZeRO-3 at nd = 1000: rank 0's shard updated, then each unit assembled from
    # 1000 shards (the gather's per-rank pointer table at its largest use), both
    # 16-bit and 8-bit quantized
    import torch
    nd = 1000
    c = H.Case(shapes=[(40_000,), (7,), (3_001, 3)], nd=nd, stage=3, units=[0, 0, 1], steps=2,
               clip=1.0)
    plans = []
    gpu = H.run_gpu(z, c, plan_out=plans)
    plan = plans[0]
    try:
        _, total, nunits, _ = z.zero_plan_layout(plan)
        assert nunits == 2
        mask = H.stage3_valid_mask(z, plan, nd)
        ora = H.run_oracle(c, total, total, mask, follow=gpu.results)
        H.compare_runs(gpu, ora, "stage3 nd=1000")
        H.assert_state_equal(gpu, ora, "stage3 nd=1000")
        dev = torch.device("cuda", 0)
        sp = torch.cuda.current_stream().cuda_stream
        host_shards = [gpu.params]
        for k in range(1, nd):
            s = gen.s16(c.seed, gen.STREAM_SHARD, 0, k, total, 0.02, 1.0, c.dtype)
            s[~H.stage3_valid_mask(z, plan, nd, rank=k)] = 0
            host_shards.append(s)
        stacked = torch.from_numpy(np.stack(host_shards).view(np.int16)).to(dev)
        shards = [stacked[k] for k in range(nd)]
        qs = [oracle.quantize_16(c.dtype, s, 8, 256) for s in host_shards]
        codes = torch.from_numpy(np.stack([q for q, _ in qs])).to(dev)
        scales = torch.from_numpy(np.stack([s for _, s in qs])).to(dev)
        for u in range(nunits):
            ln, sl, off = z.zero_plan_unit(plan, u)
            out = torch.full((ln + 8,), -1, dtype=torch.int16, device=dev)
            z.zero_gather_layer(plan, u, shards, out, sp)
            torch.cuda.synchronize()
            got = out.cpu().numpy().view(np.uint16)
            want = oracle.gather_unit(nd, ln, sl, [s[off:off + sl] for s in host_shards])
            assert np.array_equal(got[:ln], want) and np.all(got[ln:] == 0xFFFF)
            out.fill_(-1)
            z.zero_gather_layer_q(plan, u, 8, [codes[k] for k in range(nd)],
                                  [scales[k] for k in range(nd)], out, sp)
            torch.cuda.synchronize()
            got = out.cpu().numpy().view(np.uint16)
            want = oracle.gather_unit_q(c.dtype, nd, ln, sl, off, 8, 256, [q for q, _ in qs],
                                        [s for _, s in qs])
            assert np.array_equal(got[:ln], want) and np.all(got[ln:] == 0xFFFF)
    finally:
        z.zero_plan_destroy(plan)


# ---- degenerate settings of the method ----
DEGENERATE = {
    "lr-zero": dict(lr=0.0, clip=1.0),                  # master unchanged; m and v still advance
    "beta1-zero": dict(beta1=0.0, clip=1.0),            # m is the (clipped) gradient itself
    "beta2-zero": dict(beta2=0.0),                      # v is the squared gradient itself
    "clip-vanishing": dict(clip=1e-30),                 # c ~ 5e-31: the squares of the clipped gradients underflow to 0
    "l2-decay-clip": dict(weight_decay=0.5, decoupled_wd=0, clip=0.1),
    "eps-large": dict(eps=1.0, clip=1.0),
}


@pytest.mark.parametrize("name", sorted(DEGENERATE))
@pytest.mark.parametrize("kernels", [None, 0])
def test_degenerate_settings(z, name, kernels):
    # against the oracle; the two-pass kernels and the plan's own choice.  With
    # the clip on, the state is within tolerance (c may differ in its last bit);
    # without it, bit for bit.
    kw = DEGENERATE[name]
    c = H.Case(shapes=[(50_003,), (5,)], nd=4, steps=3, **kw)
    gpu, _ = check(z, c, reduce_kernel=kernels)
    if name == "lr-zero":
        master0 = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, c.psi, 0.02)
        assert gpu.master.tobytes() == master0.tobytes()
        assert np.any(gpu.m != 0) and np.any(gpu.v != 0)
    if name == "clip-vanishing":
        assert all(r["clip_coef"] < 1e-28 for r in gpu.results)


@pytest.mark.parametrize("nd", [3, 16])
@pytest.mark.parametrize("mode", ["fused", "clip", "fp16-dyn"])
def test_stage3_modes(z, nd, mode):
    # ZeRO-3 (one rank's shard resident, its nd contributions) on every kernel path,
    # with ragged units; state against the oracle, skips and scale schedule exact
    shapes, units = [(30_011,), (7,), (1_000, 13), (5,)], [0, 0, 1, 2]
    if mode == "fused":
        c = H.Case(shapes=shapes, nd=nd, stage=3, units=units, steps=3, weight_decay=0.01)
    elif mode == "clip":
        c = H.Case(shapes=shapes, nd=nd, stage=3, units=units, steps=3, clip=0.05,
                   weight_decay=0.01, decoupled_wd=0)
    else:
        c = H.Case(shapes=shapes, nd=nd, stage=3, units=units, steps=4, dtype=gen.FP16,
                   grad_sigma=1e-3, loss_scale=4096.0, dynamic_scale=1, inf_steps=(2,),
                   growth_interval=2)
    gpu, _ = check(z, c)
    if mode == "fp16-dyn":
        assert [r["skipped"] for r in gpu.results] == [0, 1, 0, 0]
