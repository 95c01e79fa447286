"""ZeRO-Offload steps on the GPU + host against the oracle ([L18] sec. 4.4; [ZL8]
sec. 6.2, 7): the device reduce writes the 16-bit averaged gradient (compared
bit for bit), the host updates master, m, v (host arrays) and the 16-bit
parameters land on the device; several steps, with an overflow skip, clipping,
weight decay, ragged sizes and more than one pipelined chunk."""
import dataclasses

import numpy as np
import pytest

import gen
import harness as H
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_sharded_mixed_02_gb300 import build
    build.build()
    import zero_sharded_mixed_02_gb300 as z
    z.lib()
    return torch, z


def run_offload(torch, z, c, nthreads=0):
    plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z))
    try:
        _, padded, _, _ = z.zero_plan_layout(plan)
        n = c.psi
        master = np.zeros(padded, np.float32)
        master[:n] = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, n, 0.02)
        m = np.zeros(padded, np.float32)
        v = np.zeros(padded, np.float32)
        params = torch.zeros(padded, dtype=torch.int16, device="cuda")
        work = torch.zeros(padded, dtype=torch.int16, device="cuda")
        grads = torch.empty((c.nd, padded), dtype=torch.int16, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        results, scale, last_g = [], c.loss_scale, None
        for step in range(1, c.steps + 1):
            g = H.grads_for_step(c, step, n, padded, scale)
            grads.copy_(torch.from_numpy(g.view(np.int16)))
            z.zero_offload_step(plan, grads, master, m, v, params, work, nthreads, stream)
            r = z.zero_step_result(plan)
            r["overflow"] = z.zero_step_overflow(plan)
            results.append(r)
            last_g = (g, scale)
            scale = r["loss_scale"]
        torch.cuda.synchronize()
        g16 = work[:n].cpu().numpy().view(np.uint16)
        out = H.Run(master[:n].copy(), m[:n].copy(), v[:n].copy(),
                    params[:n].cpu().numpy().view(np.uint16), results)
        return out, g16, last_g
    finally:
        z.zero_plan_destroy(plan)


def run_oracle_offload(c, follow=None):
    """The oracle's offloaded steps; follow: the GPU's per-step results, whose
    clip coefficients it admits (harness.admit_clip)."""
    n = c.psi
    state = [gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, n, 0.02), np.zeros(n, np.float32),
             np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    st = oracle.new_scalars(c.loss_scale)
    res = []
    for step in range(1, c.steps + 1):
        g = np.ascontiguousarray(H.grads_for_step(c, step, n, n, st.loss_scale))
        if follow is None:
            r = oracle.step_offload(c.nd, c.dtype, g, *state, c.opt(), st)
        else:
            r = H.oracle_step_admitting(c.nd, c.dtype, g, *state, c.opt(), st, follow[step - 1],
                                        offload=True, what=f"step {step}")
        r["loss_scale"] = st.loss_scale
        r["t"] = st.t
        res.append(r)
    return H.Run(*state, res)


CASES = [
    H.Case(shapes=[(3_000_001,), (77,), (1_048_576,)], nd=16, dtype=gen.FP16, grad_sigma=1e-3,
           loss_scale=65536.0, dynamic_scale=1, clip=1.0, steps=4, inf_steps=(2,)),
    H.Case(shapes=[(40_000_003,)], nd=3, clip=0.5, weight_decay=0.01, steps=2),   # 3 chunks
    H.Case(shapes=[(1000,), (24,)], nd=1, steps=2),
    H.Case(shapes=[(5000,)], nd=5, dtype=gen.FP16, grad_sigma=1e-2, loss_scale=1024.0,
           weight_decay=0.01, decoupled_wd=0, steps=2),
    # static scale with skip_on_overflow: the step with +inf skipped, nothing copied back
    H.Case(shapes=[(70_001,)], nd=4, skip_on_overflow=1, steps=4, inf_steps=(2,)),
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"nd{c.nd}-psi{c.psi}")
def test_offload_step_matches_oracle(env, c):
    torch, z = env
    gpu, g16, (g_last, s_last) = run_offload(torch, z, c)
    ora = run_oracle_offload(c, follow=gpu.results)
    H.compare_runs(gpu, ora, what="offload")
    want16, _, _ = oracle.reduce16(c.nd, c.dtype, np.ascontiguousarray(g_last[:, :c.psi]),
                                   loss_scale=s_last)
    assert np.array_equal(g16, want16)                     # the copied gradient, bit for bit
    for a, b in zip((gpu.master, gpu.m, gpu.v, gpu.params), (ora.master, ora.m, ora.v, ora.params)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    if c.inf_steps:
        assert [r["skipped"] for r in gpu.results] == [0, 1, 0, 0]


def test_thread_counts_agree(env):
    torch, z = env
    c = CASES[1]
    a, _, _ = run_offload(torch, z, dataclasses.replace(c, steps=1), nthreads=1)
    b, _, _ = run_offload(torch, z, dataclasses.replace(c, steps=1), nthreads=7)
    for x, y in zip((a.master, a.m, a.v, a.params), (b.master, b.m, b.v, b.params)):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_offload_argument_checks(env):
    torch, z = env
    c = H.Case(shapes=[(4096,)], nd=4)
    p3 = z.zero_plan_create(c.psi, c.nd, 3, c.dtype, c.shapes, c.hparams(z))
    p2 = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        h = np.zeros(4096, np.float32)
        d = torch.zeros(4 * 4096, dtype=torch.int16, device="cuda")
        with pytest.raises(z.ZeroError) as e:
            z.zero_offload_step(p3, d, h, h, h, d, d)        # stage 3
        assert e.value.code == z.ZERO_EINVAL
        with pytest.raises(z.ZeroError) as e:
            z.zero_offload_step(p2, d.data_ptr() + 2, h, h, h, d, d)
        assert e.value.code == z.ZERO_EINVAL
        with pytest.raises(z.ZeroError) as e:
            z.zero_offload_step(p2, d, None, h, h, d, d)
        assert e.value.code == z.ZERO_EINVAL
    finally:
        z.zero_plan_destroy(p3)
        z.zero_plan_destroy(p2)


def test_gpt2_small_full_size(env):
    """All 124 M parameters of the GPT-2 small list (Nd = 8, bf16, AdamW,
    clip 1.0), two offloaded steps, every element against the oracle."""
    from gen import workloads as W
    torch, z = env
    c = H.from_workload(W.gpt2_small(), steps=2)
    gpu, _, _ = run_offload(torch, z, c)
    ora = run_oracle_offload(c, follow=gpu.results)
    H.compare_runs(gpu, ora, what="GPT-2 small offload")
    H.assert_state_equal(gpu, ora, what="GPT-2 small offload")
