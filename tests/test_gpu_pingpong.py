"""zero_step_pingpong: the single-pass step with two state sets, where a step
that is not skipped makes the set it wrote current.  Against zero_step on the
same inputs, after every step: the current set's master, m, v and the 16-bit
parameters (rewritten from the current set after a skipped step) bit for bit,
the step report's skip, scale and t exactly and its norm within the harness's
tolerance (the two paths sum the squares over different grids).  Against the oracle: the results by the harness's rules and
the state bit for bit.  Schedules plant +inf and NaN so that steps are skipped."""
import numpy as np
import pytest

import gen
import harness as H

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


CASES = {
    "tiny-flat-fp16-dynamic": dict(shapes=[(512, 1024), (1024,), (1024, 512), (512,)], nd=4,
                                   dtype=gen.FP16, grad_sigma=1e-3, loss_scale=1024.0,
                                   dynamic_scale=1, growth_interval=3),
    "fp16-dynamic-nd16-ragged": dict(shapes=[(300_007,), (13,)], nd=16, dtype=gen.FP16,
                                     grad_sigma=1e-3, loss_scale=4096.0, dynamic_scale=1),
    "bf16-skip-on-overflow-nd3": dict(shapes=[(200_001,)], nd=3, skip_on_overflow=1,
                                      weight_decay=0.01),
    "fp16-dynamic-stage3-nd8": dict(shapes=[(5000,), (77,), (3000, 3)], units=[0, 0, 1], nd=8,
                                    stage=3, dtype=gen.FP16, grad_sigma=1e-3, loss_scale=2048.0,
                                    dynamic_scale=1),
}


def run_pair(torch, z, c):
    """The case's steps through zero_step_pingpong (plan A, two state sets) and
    zero_step (plan B); per step: A's current set, A's params, A's report, B's
    state and report."""
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    units = c.units if c.stage == 3 else None
    pa = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z), units=units)
    pb = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z), units=units)
    try:
        _, padded, _, ws = z.zero_plan_layout(pa)
        n = c.psi if c.stage <= 2 else padded
        mask = H.stage3_valid_mask(z, pa, c.nd) if c.stage == 3 else None
        master0 = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, n, 0.02)
        if mask is not None:
            master0[~mask] = 0

        def state_set():
            s = [torch.zeros(padded, dtype=torch.float32, device=dev) for _ in range(3)]
            s[0][:n] = torch.from_numpy(master0).to(dev)
            return s
        sets = [state_set(), [torch.full((padded,), float("nan"), device=dev) for _ in range(3)]]
        pa_params = torch.zeros(padded, dtype=torch.int16, device=dev)
        sb = state_set()
        pb_params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev) if ws else None
        grads = torch.empty((c.nd, padded), dtype=torch.int16, device=dev)
        assert z.zero_plan_state_set(pa) == 0
        out, scale = [], c.loss_scale
        for step in range(1, c.steps + 1):
            g = H.grads_for_step(c, step, n, padded, scale, mask)
            grads.copy_(torch.from_numpy(g.view(np.int16)))
            z.zero_step_pingpong(pa, grads, sets[0], sets[1], pa_params, sp)
            z.zero_step(pb, grads, *sb, pb_params, work, sp)
            ra, rb = z.zero_step_result(pa), z.zero_step_result(pb)
            ra["overflow"] = z.zero_step_overflow(pa)
            cur = z.zero_plan_state_set(pa)
            torch.cuda.synchronize()
            out.append(dict(
                cur=cur, ra=ra, rb=rb,
                a=[t[:n].cpu().numpy() for t in sets[cur]],
                a_params=pa_params[:n].cpu().numpy().view(np.uint16),
                b=[t[:n].cpu().numpy() for t in sb],
                b_params=pb_params[:n].cpu().numpy().view(np.uint16)))
            scale = ra["loss_scale"]
        return out, n, padded, mask
    finally:
        z.zero_plan_destroy(pa)
        z.zero_plan_destroy(pb)


@pytest.mark.parametrize("name", sorted(CASES))
def test_pingpong_matches_zero_step_and_the_oracle(env, name):
    torch, z = env
    c = H.Case(steps=6, inf_steps=(2,), nan_steps=(4,), **CASES[name])
    out, n, padded, mask = run_pair(torch, z, c)
    # the current set flips on every step that is not skipped
    skips = [o["ra"]["skipped"] for o in out]
    assert skips == [0, 1, 0, 1, 0, 0]
    assert [o["cur"] for o in out] == [1, 1, 0, 0, 1, 0]
    for k, o in enumerate(out, start=1):
        ra, rb = o["ra"], o["rb"]
        for key in ("skipped", "loss_scale", "t", "clip_coef"):
            assert ra[key] == rb[key], (k, key, ra, rb)
        # the two paths sum the norm's squares over different grids
        if np.isfinite(rb["grad_norm"]):
            assert abs(ra["grad_norm"] - rb["grad_norm"]) <= H.REL_NORM * rb["grad_norm"], k
        else:
            assert not np.isfinite(ra["grad_norm"]), k
        for x, y in zip(o["a"], o["b"]):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), k
        assert np.array_equal(o["a_params"], o["b_params"]), k
    # and the oracle, admitting the GPU's clip coefficient (no clip here: c = 1)
    last = out[-1]
    gpu = H.Run(*last["a"], last["a_params"], [o["ra"] for o in out])
    ora = H.run_oracle(c, n, padded, mask, follow=gpu.results)
    H.compare_runs(gpu, ora, what=name)
    H.assert_state_equal(gpu, ora, what=name)


def test_pingpong_rejects_a_clip_and_bad_pointers(env):
    torch, z = env
    t = torch.zeros(4096, dtype=torch.float32, device="cuda")
    c = H.Case(shapes=[(4096,)], nd=4, clip=1.0)
    plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_pingpong(plan, t, (t, t, t), (t, t, t), t)
        assert e.value.code == z.ZERO_EINVAL
    finally:
        z.zero_plan_destroy(plan)
    c = H.Case(shapes=[(4096,)], nd=4, dtype=gen.FP16, loss_scale=8.0, dynamic_scale=1)
    plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_pingpong(plan, t, (t, t, t), (t, None, t), t)
        assert e.value.code == z.ZERO_EINVAL
        with pytest.raises(z.ZeroError) as e:
            z.zero_step_pingpong(plan, t, (t, t, t), (t, t, t.data_ptr() + 4), t)
        assert e.value.code == z.ZERO_EINVAL
    finally:
        z.zero_plan_destroy(plan)
