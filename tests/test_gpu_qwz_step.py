"""zero_step_qwz: a ZeRO-3 step whose update pass also quantizes the updated
shard for the qwZ gather.  Against the oracle: the state after every step as
zero_step's parity rules require, and the codes and scales bit for bit equal to
the oracle's block quantizer applied to the oracle's own updated 16-bit shard.
Against zero_step on the same inputs: master, m, v and parameters bit for bit.
The code buffers are filled with garbage before the steps that matter (a
skipped step included), so every code and scale must be written by the step.

Shard layouts put partial 256-element blocks at the shard's end and blocks that
straddle unit boundaries (blocks count from the shard's start)."""
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


SMALL = dict(shapes=[(1270,), (700,), (200,)], units=[0, 1, 2])          # slices 320 + 192 + 64
LARGE = dict(shapes=[(1_000_003,), (77_777,), (3000,)], units=[0, 1, 2])

CASES = {
    # name: (case settings, kernel path)
    "fused-bf16-nd4": (dict(nd=4, dtype=gen.BF16, **SMALL), 0),
    "fused-bf16-nd4-large": (dict(nd=4, dtype=gen.BF16, **LARGE), 0),
    "fused-fp16-nd3-generic": (dict(nd=3, dtype=gen.FP16, grad_sigma=1e-3, **LARGE), 0),
    "fused-bf16-nd64": (dict(nd=64, dtype=gen.BF16, shapes=[(100_000,), (5000,)], units=[0, 1]),
                        0),
    "two-pass-bf16-nd8": (dict(nd=8, dtype=gen.BF16, skip_on_overflow=1, **LARGE), 1),
    "recompute-bf16-nd2": (dict(nd=2, dtype=gen.BF16, skip_on_overflow=1, **LARGE), 2),
    "two-pass-fp16-dynamic-skip": (dict(nd=4, dtype=gen.FP16, grad_sigma=1e-3, loss_scale=1024.0,
                                        dynamic_scale=1, inf_steps=(2,), **LARGE), 1),
    "recompute-fp16-dynamic-skip": (dict(nd=2, dtype=gen.FP16, grad_sigma=1e-3,
                                         loss_scale=1024.0, dynamic_scale=1, inf_steps=(2,),
                                         **SMALL), 2),
}


def run_both(torch, z, c, bits):
    """The same seeded steps through zero_step_qwz (plan A) and zero_step (plan
    B); returns A's codes and scales after every step and both final states."""
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    plans = [z.zero_plan_create(c.psi, c.nd, 3, c.dtype, c.shapes, c.hparams(z), units=c.units)
             for _ in range(2)]
    try:
        _, L, _, ws = z.zero_plan_layout(plans[0])
        mask = H.stage3_valid_mask(z, plans[0], c.nd)
        master0 = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, L, 0.02)
        master0[~mask] = 0
        bufs = []
        for _ in range(2):
            st = [torch.from_numpy(master0.copy()).to(dev)] + \
                 [torch.zeros(L, dtype=torch.float32, device=dev) for _ in range(2)] + \
                 [torch.zeros(L, dtype=torch.int16, device=dev)]
            work = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev) if ws else None
            bufs.append((st, work))
        nbytes = L if bits == 8 else L // 2
        codes = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        scales = torch.empty(-(-L // 256), dtype=torch.float32, device=dev)
        grads = torch.empty((c.nd, L), dtype=torch.int16, device=dev)
        per_step, scale = [], c.loss_scale
        for step in range(1, c.steps + 1):
            g = H.grads_for_step(c, step, L, L, scale, mask)
            grads.copy_(torch.from_numpy(g.view(np.int16)))
            codes.fill_(0xA5)                                    # garbage: the step writes all
            scales.fill_(float("nan"))
            (sa, wa), (sb, wb) = bufs
            z.zero_step_qwz(plans[0], grads, *sa, wa, bits, codes, scales, sp)
            z.zero_step(plans[1], grads, *sb, wb, sp)
            ra, rb = z.zero_step_result(plans[0]), z.zero_step_result(plans[1])
            assert ra == rb, (step, ra, rb)
            per_step.append((codes.cpu().numpy(), scales.cpu().numpy(), ra))
            scale = ra["loss_scale"]
        torch.cuda.synchronize()
        out = [[t.cpu().numpy() for t in st] for st, _ in bufs]
        for o in out:
            o[3] = o[3].view(np.uint16)
        return per_step, out, L, mask
    finally:
        for p in plans:
            z.zero_plan_destroy(p)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("name", sorted(CASES))
def test_step_qwz_against_oracle_and_zero_step(env, name, bits):
    torch, z = env
    over, path = CASES[name]
    c = H.Case(steps=3, stage=3, **over)
    plan = z.zero_plan_create(c.psi, c.nd, 3, c.dtype, c.shapes, c.hparams(z), units=c.units)
    assert z.zero_plan_path(plan) == path
    z.zero_plan_destroy(plan)
    per_step, (qa, qb), L, mask = run_both(torch, z, c, bits)
    # zero_step and zero_step_qwz leave the same state, bit for bit
    for x, y in zip(qa, qb):
        assert np.array_equal(x.view(np.uint32 if x.dtype == np.float32 else np.uint16),
                              y.view(np.uint32 if y.dtype == np.float32 else np.uint16))
    # the oracle, step by step: its state, then its quantizer on its own shard
    master = gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, L, 0.02)
    master[~mask] = 0
    m, v, params = np.zeros(L, np.float32), np.zeros(L, np.float32), np.zeros(L, np.uint16)
    st = oracle.new_scalars(c.loss_scale)
    skips = []
    for step, (codes, scales, res) in enumerate(per_step, start=1):
        g = H.grads_for_step(c, step, L, L, st.loss_scale, mask)
        r = oracle.step(c.nd, c.dtype, np.ascontiguousarray(g), master, m, v, params, c.opt(), st)
        assert r["skipped"] == res["skipped"]
        skips.append(r["skipped"])
        q, s = oracle.quantize_16(c.dtype, params, bits, 256)
        assert np.array_equal(scales.view(np.uint32), s.view(np.uint32)), f"step {step} scales"
        assert np.array_equal(codes, q), f"step {step} codes"
    if c.inf_steps:
        assert skips == [0, 1, 0]
    H.assert_state_close(qa, (master, m, v, params), name)


@pytest.mark.parametrize("bits", [8, 4])
def test_step_qwz_with_clip_matches_the_standalone_quantizer(env, bits):
    """With a clip, the oracle admits the GPU's clip coefficient (the harness's
    rule); the state is then the oracle's bit for bit, and the codes are checked
    against zero_quantize_shard of the same updated shard and against the
    oracle's quantizer on the oracle's shard."""
    torch, z = env
    c = H.Case(steps=3, stage=3, nd=8, dtype=gen.BF16, clip=0.05, **LARGE)
    per_step, (qa, _), L, mask = run_both(torch, z, c, bits)
    d = torch.from_numpy(qa[3].view(np.int16)).cuda()
    codes = torch.empty(L if bits == 8 else L // 2, dtype=torch.uint8, device="cuda")
    scales = torch.empty(-(-L // 256), dtype=torch.float32, device="cuda")
    z.zero_quantize_shard(c.dtype, d, L, bits, codes, scales,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(per_step[-1][0], codes.cpu().numpy())
    assert np.array_equal(per_step[-1][1].view(np.uint32), scales.cpu().numpy().view(np.uint32))
    ora = H.run_oracle(c, L, L, mask, follow=[r for _, _, r in per_step])
    H.assert_state_equal(H.Run(*qa, []), ora, "clip")
    q, s = oracle.quantize_16(c.dtype, ora.params, bits, 256)
    assert np.array_equal(per_step[-1][0], q)
    assert np.array_equal(per_step[-1][1].view(np.uint32), s.view(np.uint32))


def test_step_qwz_rejects_bad_arguments(env):
    torch, z = env
    c = H.Case(stage=3, nd=4, **SMALL)
    t = torch.zeros(4096, dtype=torch.float32, device="cuda")
    plan2 = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    plan3 = z.zero_plan_create(c.psi, c.nd, 3, c.dtype, c.shapes, c.hparams(z), units=c.units)
    try:
        for plan, bits, codes in ((plan2, 8, t), (plan3, 5, t), (plan3, 8, None),
                                  (plan3, 8, t.data_ptr() + 4)):
            with pytest.raises(z.ZeroError) as e:
                z.zero_step_qwz(plan, t, t, t, t, t, None, bits, codes, t)
            assert e.value.code == z.ZERO_EINVAL
    finally:
        z.zero_plan_destroy(plan2)
        z.zero_plan_destroy(plan3)
