"""zero_grad_norm_noalloc -- the gradient norm and overflow flag for callers that
may not allocate device memory -- against the oracle (its rank-order reduce and
its binary64 sum of squares, taken on the same gradients) and against what
zero_step reports, for two calls in a row (the second reuses the library's fixed
scratch array, with a different size and different data).

This file is collected last so a stop-at-first-failure run has already run every
other test; it also passes on its own in a fresh process."""
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


def existing_entry_point(torch, z, grads_host, nd, psi, dtype, scale):
    """grad_norm and overflow as zero_step reports them (a plan with clipping, so
    the norm is computed)."""
    hp = z.hparams(clip_norm=1.0, loss_scale=scale, dynamic_scale=int(dtype == gen.FP16))
    plan = z.zero_plan_create(psi, nd, 2, dtype, [(psi,)], hp)
    try:
        _, padded, _, ws = z.zero_plan_layout(plan)
        dev = torch.device("cuda", 0)
        g = torch.from_numpy(grads_host.view(np.int16)).to(dev)
        f = [torch.zeros(padded, dtype=torch.float32, device=dev) for _ in range(3)]
        p = torch.zeros(padded, dtype=torch.int16, device=dev)
        w = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev) if ws else None
        z.zero_step(plan, g, f[0], f[1], f[2], p, w, torch.cuda.current_stream().cuda_stream)
        return z.zero_step_result(plan)["grad_norm"], z.zero_step_overflow(plan)
    finally:
        z.zero_plan_destroy(plan)


def noalloc(torch, z, grads_host, nd, psi, rank_stride, dtype, scale):
    dev = torch.device("cuda", 0)
    g = torch.from_numpy(grads_host.view(np.int16)).to(dev)
    norm = torch.full((1,), -1.0, dtype=torch.float64, device=dev)
    ovf = torch.full((1,), -1, dtype=torch.int32, device=dev)
    z.zero_grad_norm_noalloc(g, nd, psi, rank_stride, dtype, scale, norm, ovf,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return float(norm.item()), int(ovf.item())


def oracle_norm(g, nd, psi, dtype, scale):
    """The oracle's norm and flag: its reduce of the first psi elements of every
    rank's row, then the square root of its binary64 sum of squares."""
    gr, ovf = oracle.reduce(nd, dtype, np.ascontiguousarray(g[:, :psi]), loss_scale=scale)
    return float(np.sqrt(oracle.sumsq(gr))), int(ovf)


def grads(nd, psi, dtype, sigma, scale, step, inf=False):
    padded = (-(-psi // nd) + 63) // 64 * 64 * nd
    g = gen.ranks_16(0, gen.STREAM_GRAD, step, nd, psi, sigma, scale, dtype, rank_stride=padded)
    if inf:
        r, i = gen.inf_site(0, step, psi, nd)
        g[r, i] = 0x7C00 if dtype == gen.FP16 else 0x7F80
    return g, padded


@pytest.mark.parametrize("nd,dtype,sigma,scale,sizes", [
    (16, gen.FP16, 1e-3, 1024.0, (1_000_003, 262_147)),
    (3, gen.BF16, 1e-2, 1.0, (300_001, 9)),
])
def test_two_calls_in_a_row_match_zero_step(env, nd, dtype, sigma, scale, sizes):
    torch, z = env
    for call, psi in enumerate(sizes, start=1):
        g, padded = grads(nd, psi, dtype, sigma, scale, step=call)
        want_norm, want_ovf = existing_entry_point(torch, z, g, nd, psi, dtype, scale)
        got_norm, got_ovf = noalloc(torch, z, g, nd, psi, padded, dtype, scale)
        ora_norm, ora_ovf = oracle_norm(g, nd, psi, dtype, scale)
        assert got_ovf == ora_ovf == want_ovf == 0
        assert abs(got_norm - ora_norm) <= H.REL_NORM * ora_norm, (call, got_norm, ora_norm)
        assert abs(got_norm - want_norm) <= H.REL_NORM * want_norm, (call, got_norm, want_norm)


def test_overflow_flag_then_clean_call(env):
    torch, z = env
    nd, psi = 8, 500_001
    g, padded = grads(nd, psi, gen.FP16, 1e-3, 1024.0, step=3, inf=True)
    want_norm, want_ovf = existing_entry_point(torch, z, g, nd, psi, gen.FP16, 1024.0)
    got_norm, got_ovf = noalloc(torch, z, g, nd, psi, padded, gen.FP16, 1024.0)
    ora_norm, ora_ovf = oracle_norm(g, nd, psi, gen.FP16, 1024.0)
    assert got_ovf == ora_ovf == want_ovf == 1
    assert not np.isfinite(got_norm) and not np.isfinite(ora_norm)
    assert not np.isfinite(want_norm)
    g, padded = grads(nd, psi, gen.FP16, 1e-3, 1024.0, step=4)        # the flag must not stick
    want_norm, _ = existing_entry_point(torch, z, g, nd, psi, gen.FP16, 1024.0)
    got_norm, got_ovf = noalloc(torch, z, g, nd, psi, padded, gen.FP16, 1024.0)
    ora_norm, ora_ovf = oracle_norm(g, nd, psi, gen.FP16, 1024.0)
    assert got_ovf == ora_ovf == 0
    assert abs(got_norm - ora_norm) <= H.REL_NORM * ora_norm
    assert abs(got_norm - want_norm) <= H.REL_NORM * want_norm


def test_calls_take_no_device_memory(env):
    """After one call per 16-bit format (which may load the kernels and the scratch
    array's module on first use), further calls leave the device's free memory
    unchanged: the entry point allocates nothing (any device allocation takes at
    least a page of the device's free memory)."""
    torch, z = env
    dev = torch.device("cuda", 0)
    nd, psi = 4, 600_001
    bufs = {}
    for dtype in (gen.FP16, gen.BF16):
        g, padded = grads(nd, psi, dtype, 1e-3, 64.0, step=5)
        bufs[dtype] = (torch.from_numpy(g.view(np.int16)).to(dev), padded)
    norm = torch.zeros(1, dtype=torch.float64, device=dev)
    ovf = torch.zeros(1, dtype=torch.int32, device=dev)
    sp = torch.cuda.current_stream().cuda_stream
    for dtype, (g, padded) in bufs.items():                 # first calls: lazy loading
        z.zero_grad_norm_noalloc(g, nd, psi, padded, dtype, 64.0, norm, ovf, sp)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(20):
        for dtype, (g, padded) in bufs.items():
            z.zero_grad_norm_noalloc(g, nd, psi, padded, dtype, 64.0, norm, ovf, sp)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_sizes_beyond_the_scratch_are_rejected(env):
    torch, z = env
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    with pytest.raises(z.ZeroError) as e:
        z.zero_grad_norm_noalloc(out, 4, (1 << 31) + 8, (1 << 31) + 8, gen.BF16, 1.0, out,
                                 out.data_ptr() + 8)
    assert e.value.code == z.ZERO_EINVAL
