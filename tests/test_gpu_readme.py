"""The README's usage example, run as written with concrete sizes: a plan, one
step through the binding, the step's result, and the plan freed."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_readme_example_runs():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from zero_sharded_mixed_02_gb300 import build
    build.build()
    import zero_sharded_mixed_02_gb300 as z

    shapes = [(1000, 64), (64,)]
    psi, nd = 64_064, 4
    hp = z.hparams(lr=1e-3, clip_norm=1.0, loss_scale=65536.0, dynamic_scale=1)
    plan = z.zero_plan_create(psi, nd, 2, z.ZERO_FP16, shapes, hp)
    shard, padded, _, ws = z.zero_plan_layout(plan)
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(0)
    g = (rng.standard_normal((nd, padded)) * 1e-3 * 65536.0).astype(np.float16)
    g[:, psi:] = 0
    grads = torch.from_numpy(g.view(np.int16)).to(dev)
    master = torch.zeros(padded, dtype=torch.float32, device=dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    params = torch.zeros(padded, dtype=torch.int16, device=dev)
    work = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
    z.zero_step(plan, grads, master, m, v, params, work, torch.cuda.current_stream().cuda_stream)
    r = z.zero_step_result(plan)
    z.zero_plan_destroy(plan)
    assert set(r) >= {"skipped", "grad_norm", "clip_coef", "loss_scale", "t"}
    assert r["skipped"] == 0 and r["t"] == 1 and r["loss_scale"] == 65536.0
    assert np.isfinite(r["grad_norm"]) and r["grad_norm"] > 0
    assert torch.count_nonzero(master[:psi]).item() > 0        # the step moved the weights
