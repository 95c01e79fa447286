"""Parity at the full workload sizes, in the launch configuration the benchmark
times (default kernels, same plans).  Where the oracle cannot hold a whole
workload it follows sampled elements exactly (the update is elementwise) and
computes the one global quantity, the gradient norm, by streaming every
gradient through its reduce in chunks.  Inputs on the device come from the
CUDA twin of the generator, which writes the same bits as the host version."""
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
    gen.build_cuda()
    import zero_sharded_mixed_02_gb300 as z
    z.lib()
    return z


def hp_of(z, w):
    return z.hparams(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                     weight_decay=w.weight_decay, decoupled_wd=w.decoupled_wd, clip_norm=w.clip,
                     loss_scale=w.loss_scale, dynamic_scale=w.dynamic_scale, backoff=0.5,
                     growth_interval=1000)


def opt_of(w):
    return oracle.Opt(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                      weight_decay=w.weight_decay, decoupled_wd=w.decoupled_wd, clip_norm=w.clip,
                      dynamic_scale=w.dynamic_scale, backoff=0.5, growth_interval=1000)


def at(t, idx_t):
    return t.index_select(0, idx_t).cpu().numpy()


def test_gpt2_1p5b_nd16_full_schedule(z):
    """GPT-2 1.5B, Nd = 16, ZeRO-2, fp16 x65536 dynamic, clip 1.0 -- the bench
    workload at its own schedule: 10 steps, +inf planted at steps 3 and 7, so
    those two are skipped and the scale goes 65536 -> 32768 -> 16384 (each step's
    gradients generated at the scale in force).  Every non-skipped step's global
    norm is the oracle's, streamed over all 25 G gradient values; the sampled
    elements (65 K plus every shard boundary) follow all 10 steps."""
    import torch
    w = W.gpt2_xl()
    assert (w.steps, tuple(w.inf_steps)) == (10, (3, 7))
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    plan = z.zero_plan_create(w.psi, w.nd, w.stage, w.dtype, w.shapes, hp_of(z, w))
    try:
        shard, padded, _, ws = z.zero_plan_layout(plan)
        grads = torch.empty((w.nd, padded), dtype=torch.int16, device=dev)
        master = torch.zeros(padded, dtype=torch.float32, device=dev)
        m = torch.zeros_like(master)
        v = torch.zeros_like(master)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(ws // 4, dtype=torch.float32, device=dev)
        gen.cuda_f32(master.data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, w.psi, w.master_sigma,
                     cuda_stream=sp)
        idx = H.sample_indices(w.psi, shard, w.nd)
        idx_t = torch.from_numpy(idx).to(dev)
        ms = gen.f32_at(w.seed, gen.STREAM_MASTER, 0, 0, idx, w.master_sigma)
        mm, vs = np.zeros_like(ms), np.zeros_like(ms)
        ps = np.zeros(idx.size, np.uint16)
        st, opt, scale = oracle.new_scalars(w.loss_scale), opt_of(w), w.loss_scale
        skips = []
        for step in range(1, w.steps + 1):
            inject = step in w.inf_steps
            site = gen.inf_site(w.seed, step, w.psi, w.nd) if inject else None
            gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, step, w.nd, w.psi,
                              w.grad_sigma, scale, w.dtype, rank_stride=padded, cuda_stream=sp)
            if site:
                grads[site[0], site[1]] = 0x7C00
            z.zero_step(plan, grads, master, m, v, params, work, sp)
            r = z.zero_step_result(plan)
            if inject:
                # the planted +inf is the only non-finite input: the oracle's flag is set
                g16 = H.oracle_sampled_grads(w.seed, step, w.nd, np.array([site[1]]), w.grad_sigma,
                                             scale, w.dtype, inf_at=site)
                _, ovf = oracle.reduce(w.nd, w.dtype, g16, loss_scale=scale)
                assert ovf
                norm = float("inf")
            else:
                norm, ovf = H.oracle_norm_streamed(w.seed, step, w.nd, w.psi, w.grad_sigma,
                                                   scale, w.dtype)
                assert not ovf
            c = oracle.clip_coef(norm, w.clip)
            res = oracle.advance(opt, st, ovf)
            if not res.skipped:
                c_used = H.admit_clip(c, r, f"step {step}")
            skips.append(r["skipped"])
            assert r["skipped"] == res.skipped == int(inject), f"step {step}"
            assert z.zero_step_overflow(plan) == int(ovf)
            assert (r["t"], r["loss_scale"]) == (st.t, st.loss_scale), f"step {step}"
            if not res.skipped:
                assert abs(r["grad_norm"] - norm) <= H.REL_NORM * norm, f"step {step}"
                assert H.ulps32(r["clip_coef"], c) <= H.CLIP_ULPS, f"step {step}"
                g16 = H.oracle_sampled_grads(w.seed, step, w.nd, idx, w.grad_sigma, scale, w.dtype)
                g, _ = oracle.reduce(w.nd, w.dtype, g16, loss_scale=scale)
                # the reduced gradient in the workspace is bit-exact at every sample
                assert np.array_equal(at(work, idx_t).view(np.uint32), g.view(np.uint32))
                oracle.adam(g, c_used, ms, mm, vs, ps, w.dtype, opt, res.bc1, res.bc2)
            else:
                assert not np.isfinite(r["grad_norm"])
            for x, y in zip((at(master, idx_t), at(m, idx_t), at(v, idx_t)), (ms, mm, vs)):
                assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), f"step {step}"
            assert np.array_equal(at(params, idx_t).view(np.uint16), ps), f"step {step}"
            scale = st.loss_scale
        assert skips == [0, 0, 1, 0, 0, 0, 1, 0, 0, 0]
        assert (st.t, st.loss_scale) == (8, 16384.0)
    finally:
        z.zero_plan_destroy(plan)


def test_gpt2_small_nd8_full_size_all_elements(z):
    """GPT-2 small, Nd = 8, ZeRO-1, bf16, AdamW 0.01, clip 1.0, 10 steps: every
    element of every output bit for bit against the oracle (which admits the
    GPU's clip coefficient when it is within the harness's bound of its own)."""
    import torch
    w = W.gpt2_small()
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    plan = z.zero_plan_create(w.psi, w.nd, w.stage, w.dtype, w.shapes, hp_of(z, w))
    try:
        _, padded, _, ws = z.zero_plan_layout(plan)
        grads = torch.empty((w.nd, padded), dtype=torch.int16, device=dev)
        master = torch.zeros(padded, dtype=torch.float32, device=dev)
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(ws // 4, dtype=torch.float32, device=dev)
        gen.cuda_f32(master.data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, w.psi, w.master_sigma,
                     cuda_stream=sp)
        om = gen.f32(w.seed, gen.STREAM_MASTER, 0, 0, w.psi, w.master_sigma)
        omm, ov = np.zeros_like(om), np.zeros_like(om)
        op = np.zeros(w.psi, np.uint16)
        st, opt = oracle.new_scalars(w.loss_scale), opt_of(w)
        for step in range(1, w.steps + 1):
            gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, step, w.nd, w.psi,
                              w.grad_sigma, 1.0, w.dtype, rank_stride=padded, cuda_stream=sp)
            z.zero_step(plan, grads, master, m, v, params, work, sp)
            r = z.zero_step_result(plan)
            g16 = gen.ranks_16_mt(w.seed, gen.STREAM_GRAD, step, w.nd, w.psi, w.grad_sigma, 1.0,
                                  w.dtype)
            ro = H.oracle_step_admitting(w.nd, w.dtype, g16, om, omm, ov, op, opt, st, r,
                                         what=f"step {step}")
            del g16
            assert r["t"] == st.t and r["skipped"] == ro["skipped"] == 0
            assert abs(r["grad_norm"] - ro["grad_norm"]) <= H.REL_NORM * ro["grad_norm"]
            assert r["clip_coef"] < 1.0
        torch.cuda.synchronize()
        H.assert_state_equal(H.Run(master[:w.psi].cpu().numpy(), m[:w.psi].cpu().numpy(),
                                   v[:w.psi].cpu().numpy(),
                                   params[:w.psi].cpu().numpy().view(np.uint16), []),
                             H.Run(om, omm, ov, op, []), "gpt2-small")
    finally:
        z.zero_plan_destroy(plan)


def test_llama3_8b_nd64_stage3_full_size(z):
    """LLaMA-3-8B, Nd = 64, ZeRO-3: rank 0's shard (125.5 M elements) updated
    from its 64 contributions (sampled against the oracle), then every one of
    the 34 units (embedding, 32 transformer layers, final norm + head) gathered
    from the 64 shards and compared in full with the oracle's concatenation:
    rank 0's slice of each unit from the oracle's step on that slice, ranks
    1-63's slices from the seeded shard generator."""
    import torch
    w = W.llama3_8b()
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    plan = z.zero_plan_create(w.psi, w.nd, 3, w.dtype, w.shapes, hp_of(z, w), units=w.units)
    try:
        _, total, nunits, ws = z.zero_plan_layout(plan)
        assert (total, nunits, ws) == (125_472_832, 34, 0)
        assert H.stage3_valid_mask(z, plan, w.nd).all()
        grads = torch.empty((w.nd, total), dtype=torch.int16, device=dev)
        master = torch.zeros(total, dtype=torch.float32, device=dev)
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        params = torch.zeros(total, dtype=torch.int16, device=dev)
        gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, 1, w.nd, total, w.grad_sigma,
                          1.0, w.dtype, cuda_stream=sp)
        gen.cuda_f32(master.data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, total, w.master_sigma,
                     cuda_stream=sp)
        z.zero_step(plan, grads, master, m, v, params, None, sp)
        r = z.zero_step_result(plan)
        assert r["t"] == 1 and r["skipped"] == 0
        del grads
        # sampled update of the resident shard
        idx = H.sample_indices(total, total // 64, 64)
        idx_t = torch.from_numpy(idx).to(dev)
        g16 = H.oracle_sampled_grads(w.seed, 1, w.nd, idx, w.grad_sigma, 1.0, w.dtype)
        ms = gen.f32_at(w.seed, gen.STREAM_MASTER, 0, 0, idx, w.master_sigma)
        mm, vs, ps = np.zeros_like(ms), np.zeros_like(ms), np.zeros(idx.size, np.uint16)
        oracle.step(w.nd, w.dtype, g16, ms, mm, vs, ps, opt_of(w), oracle.new_scalars())
        H.assert_state_close((at(master, idx_t), at(m, idx_t), at(v, idx_t),
                              at(params, idx_t).view(np.uint16)), (ms, mm, vs, ps), "llama rank0")
        # the other 63 ranks' parameter shards
        shards = [params]
        for k in range(1, w.nd):
            s = torch.empty(total, dtype=torch.int16, device=dev)
            gen.cuda_s16(s.data_ptr(), w.seed, gen.STREAM_SHARD, 0, k, total, w.master_sigma, 1.0,
                         w.dtype, cuda_stream=sp)
            shards.append(s)
        # every unit, every element, against the oracle
        for u in range(nunits):
            ln, sl, off = z.zero_plan_unit(plan, u)
            out = torch.empty(ln, dtype=torch.int16, device=dev)
            z.zero_gather_layer(plan, u, shards, out, sp)
            g16 = gen.ranks_16_mt(w.seed, gen.STREAM_GRAD, 1, w.nd, sl, w.grad_sigma, 1.0,
                                  w.dtype, index0=off)
            om = gen.f32(w.seed, gen.STREAM_MASTER, 0, 0, sl, w.master_sigma, index0=off)
            r0 = np.zeros(sl, np.uint16)
            oracle.step_sharded(w.nd, w.dtype, g16, om, np.zeros_like(om), np.zeros_like(om), r0,
                                opt_of(w), oracle.new_scalars(), nthreads=16)
            del g16, om
            slices = gen.ranks_16_mt(w.seed, gen.STREAM_SHARD, 0, w.nd, sl, w.master_sigma, 1.0,
                                     w.dtype, index0=off)
            slices[0] = r0
            want = oracle.gather_unit(w.nd, ln, sl, list(slices))
            del slices
            got = out.cpu().numpy().view(np.uint16)
            assert np.array_equal(got, want), f"unit {u}"   # no clip: the update is bit-exact
            del out, got, want
    finally:
        z.zero_plan_destroy(plan)


SWEEP = [(psi, nd) for psi in W.SWEEP_PSI for nd in W.SWEEP_ND]


@pytest.mark.parametrize("psi,nd", SWEEP)
def test_sweep_point_full_size(z, psi, nd):
    """Bandwidth-sweep point (flat bf16 model, ZeRO-2, no clip: the fused single
    pass), 5 warm-up steps + 1; sampled elements followed through all 6 steps."""
    import torch
    w = W.sweep(psi, nd)
    dev = torch.device("cuda", 0)
    sp = torch.cuda.current_stream().cuda_stream
    torch.cuda.empty_cache()                 # earlier tests' cached blocks
    free = torch.cuda.mem_get_info()[0]
    need = 2 * nd * psi + 14 * psi + (1 << 30)
    if need > free:
        pytest.skip(f"needs {need / 1e9:.0f} GB, {free / 1e9:.0f} GB free")
    plan = z.zero_plan_create(w.psi, w.nd, w.stage, w.dtype, w.shapes, hp_of(z, w))
    try:
        shard, padded, _, ws = z.zero_plan_layout(plan)
        assert ws == 0 and z.zero_plan_path(plan) == z.PATH_FUSED
        grads = torch.empty((nd, padded), dtype=torch.int16, device=dev)
        master = torch.zeros(padded, dtype=torch.float32, device=dev)
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        gen.cuda_f32(master.data_ptr(), w.seed, gen.STREAM_MASTER, 0, 0, psi, w.master_sigma,
                     cuda_stream=sp)
        idx = H.sample_indices(psi, shard, nd, k=1 << 14)
        idx_t = torch.from_numpy(idx).to(dev)
        ms = gen.f32_at(w.seed, gen.STREAM_MASTER, 0, 0, idx, w.master_sigma)
        mm, vs, ps = np.zeros_like(ms), np.zeros_like(ms), np.zeros(idx.size, np.uint16)
        st = oracle.new_scalars()
        for step in range(1, w.steps + 1):
            gen.cuda_ranks_16(grads.data_ptr(), w.seed, gen.STREAM_GRAD, step, nd, psi,
                              w.grad_sigma, 1.0, w.dtype, rank_stride=padded, cuda_stream=sp)
            z.zero_step(plan, grads, master, m, v, params, None, sp)
            g16 = H.oracle_sampled_grads(w.seed, step, nd, idx, w.grad_sigma, 1.0, w.dtype)
            oracle.step(nd, w.dtype, g16, ms, mm, vs, ps, opt_of(w), st)
        assert z.zero_step_result(plan)["t"] == w.steps
        for x, y in zip((at(master, idx_t), at(m, idx_t), at(v, idx_t)), (ms, mm, vs)):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))   # no clip: bit-exact
        assert np.array_equal(at(params, idx_t).view(np.uint16), ps)
    finally:
        z.zero_plan_destroy(plan)
