"""Bucketed steps (constant-size gradient buckets): a synthetic backward pass on
one stream writes each bucket's nd gradient contributions into one of two
bucket buffers, in reverse bucket order (the backward pass reaches the last
layers first); the bucket reduces follow on another stream; then the update.
Checked against the oracle's unbucketed step on the same inputs."""
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
    gen.build_cuda()
    import zero_sharded_mixed_02_gb300 as z
    z.lib()
    return torch, z


def run_bucketed(torch, z, c, bucket_elems, reverse=True):
    dev = torch.device("cuda", 0)
    plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z))
    try:
        ws = z.zero_plan_set_bucket(plan, bucket_elems)
        n = c.psi
        _, padded, _, _ = z.zero_plan_layout(plan)
        nb = -(-n // bucket_elems)
        master = torch.zeros(padded, dtype=torch.float32, device=dev)
        master[:n] = torch.from_numpy(gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, n, 0.02)).to(dev)
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        params = torch.zeros(padded, dtype=torch.int16, device=dev)
        work = torch.empty(ws // 4, dtype=torch.float32, device=dev)
        bufs = [torch.empty((c.nd, bucket_elems), dtype=torch.int16, device=dev) for _ in range(2)]
        producer, consumer = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        freed = [None, None]
        results, scale = [], c.loss_scale
        order = list(range(nb))[::-1] if reverse else list(range(nb))
        for step in range(1, c.steps + 1):
            # +inf / NaN at the same site harness.grads_for_step plants them
            bits = (0x7C00 if c.dtype == gen.FP16 else 0x7F80) if step in c.inf_steps else \
                   (0x7E00 if c.dtype == gen.FP16 else 0x7FC0) if step in c.nan_steps else None
            site = gen.inf_site(c.seed, step, n, c.nd) if bits is not None else None
            for j, b in enumerate(order):
                buf = bufs[j % 2]
                first, count = b * bucket_elems, min(bucket_elems, n - b * bucket_elems)
                with torch.cuda.stream(producer):
                    if freed[j % 2] is not None:
                        producer.wait_event(freed[j % 2])
                    gen.cuda_ranks_16(buf.data_ptr(), c.seed, gen.STREAM_GRAD, step, c.nd, count,
                                      c.grad_sigma, scale, c.dtype, rank_stride=bucket_elems,
                                      index0=first, cuda_stream=producer.cuda_stream)
                    if site and first <= site[1] < first + count:
                        buf[site[0], site[1] - first] = bits
                    ready = torch.cuda.Event()
                    ready.record(producer)
                consumer.wait_event(ready)
                z.zero_step_bucket(plan, b, buf, work, consumer.cuda_stream)
                done = torch.cuda.Event()
                done.record(consumer)
                freed[j % 2] = done
            z.zero_step_apply(plan, master, m, v, params, work, consumer.cuda_stream)
            r = z.zero_step_result(plan)
            r["overflow"] = z.zero_step_overflow(plan)
            results.append(r)
            scale = r["loss_scale"]
        torch.cuda.synchronize()
        return H.Run(master[:n].cpu().numpy(), m[:n].cpu().numpy(), v[:n].cpu().numpy(),
                     params[:n].cpu().numpy().view(np.uint16), results,
                     g32=work[:n].cpu().numpy()), padded
    finally:
        z.zero_plan_destroy(plan)


CASES = [
    (H.Case(shapes=[(1_000_003,)], nd=16, dtype=gen.FP16, grad_sigma=1e-3, loss_scale=65536.0,
            dynamic_scale=1, clip=1.0, steps=4, inf_steps=(2,)), 1 << 17),
    (H.Case(shapes=[(300_001,), (77,)], nd=3, clip=0.5, steps=3, weight_decay=0.01), 65536),
    (H.Case(shapes=[(1 << 20,)], nd=8, steps=3), 1 << 20),            # one bucket
    (H.Case(shapes=[(5000,)], nd=4, clip=1.0, steps=2), 64),         # many tiny buckets
    # static scale with skip_on_overflow: +inf at step 2 and NaN at step 3 both skip
    (H.Case(shapes=[(200_003,)], nd=8, skip_on_overflow=1, steps=4, inf_steps=(2,),
            nan_steps=(3,)), 32768),
]


@pytest.mark.parametrize("case,bucket", CASES)
@pytest.mark.parametrize("reverse", [True, False])
def test_bucketed_step_matches_oracle(env, case, bucket, reverse):
    torch, z = env
    gpu, padded = run_bucketed(torch, z, case, bucket, reverse)
    ora = H.run_oracle(case, case.psi, padded, follow=gpu.results)
    H.compare_runs(gpu, ora, what=f"bucket={bucket}")
    H.assert_state_equal(gpu, ora, what=f"bucket={bucket}")
    # the reduced gradient of the last step, bit for bit
    last = case.steps
    scale = gpu.results[-2]["loss_scale"] if last > 1 else case.loss_scale
    g = H.grads_for_step(case, last, case.psi, case.psi, scale)
    import oracle
    want, _ = oracle.reduce(case.nd, case.dtype, g, loss_scale=scale)
    assert np.array_equal(gpu.g32.view(np.uint32), want.view(np.uint32))


def test_bucket_contract_errors(env):
    torch, z = env
    c = H.Case(shapes=[(4096,)], nd=4, clip=1.0)
    plan = z.zero_plan_create(c.psi, c.nd, 2, c.dtype, c.shapes, c.hparams(z))
    try:
        with pytest.raises(z.ZeroError):
            z.zero_plan_set_bucket(plan, 100)                    # not a multiple of 64
        ws = z.zero_plan_set_bucket(plan, 1024)
        work = torch.zeros(ws // 4, dtype=torch.float32, device="cuda")
        buf = torch.zeros((4, 1024), dtype=torch.int16, device="cuda")
        st = [torch.zeros(4096, dtype=torch.float32, device="cuda") for _ in range(3)]
        p = torch.zeros(4096, dtype=torch.int16, device="cuda")
        with pytest.raises(z.ZeroError):
            z.zero_step_bucket(plan, 4, buf, work)                # bucket out of range
        z.zero_step_bucket(plan, 0, buf, work)
        with pytest.raises(z.ZeroError):
            z.zero_step_bucket(plan, 0, buf, work)                # the same bucket twice
        with pytest.raises(z.ZeroError):
            z.zero_step_apply(plan, *st, p, work)                 # buckets 1-3 missing
        for b in (3, 1, 2):
            z.zero_step_bucket(plan, b, buf, work)
        z.zero_step_apply(plan, *st, p, work)
        assert z.zero_step_result(plan)["t"] == 1
        assert z.zero_plan_set_bucket(plan, 0) == 0               # off again
        with pytest.raises(z.ZeroError):
            z.zero_step_bucket(plan, 0, buf, work)
    finally:
        z.zero_plan_destroy(plan)
