"""The parity harness's composed oracle step: with no GPU result to follow it is
the oracle's own step (zo_step, zo_step_offload) bit for bit, so admitting a
GPU clip coefficient changes nothing but that coefficient; and the admission
bound holds at exactly CLIP_ULPS units in the last place."""
import numpy as np
import pytest

import gen
import harness as H
import oracle


def _state(n, seed):
    rng = np.random.default_rng(seed)
    return [(rng.standard_normal(n) * 0.02).astype(np.float32), np.zeros(n, np.float32),
            np.zeros(n, np.float32), np.zeros(n, np.uint16)]


@pytest.mark.parametrize("offload", [False, True])
@pytest.mark.parametrize("kw", [
    dict(dtype=gen.FP16, grad_sigma=1e-3, loss_scale=1024.0, dynamic_scale=1, clip=0.05,
         inf_steps=(2,)),
    dict(dtype=gen.BF16, clip=0.05, weight_decay=0.5, decoupled_wd=0),
    dict(dtype=gen.BF16, weight_decay=0.01),
])
def test_composed_step_is_the_oracles_step(oracle, offload, kw):
    c = H.Case(shapes=[(3001,)], nd=3, steps=4, **kw)
    a, b = _state(c.psi, 1), _state(c.psi, 1)
    sa, sb = oracle.new_scalars(c.loss_scale), oracle.new_scalars(c.loss_scale)
    for step in range(1, c.steps + 1):
        g = np.ascontiguousarray(H.grads_for_step(c, step, c.psi, c.psi, sa.loss_scale))
        ra = (oracle.step_offload if offload else oracle.step)(c.nd, c.dtype, g, *a, c.opt(), sa)
        rb = H.oracle_step_admitting(c.nd, c.dtype, g, *b, c.opt(), sb, None, offload=offload)
        for k in ("skipped", "overflow", "clip_coef", "bc1", "bc2"):
            assert ra[k] == rb[k], (step, k)
        assert ra["grad_norm"] == rb["grad_norm"] or not np.isfinite(ra["grad_norm"])
        for x, y in zip(a, b):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
        assert (sa.t, sa.loss_scale) == (sb.t, sb.loss_scale)


def test_admission_bound():
    c = np.float32(0.0384529)
    up = c
    for _ in range(H.CLIP_ULPS):
        up = np.nextafter(up, np.float32(1))
    assert H.ulps32(up, c) == H.CLIP_ULPS
    assert H.admit_clip(float(c), {"clip_coef": float(up)}) == float(up)
    assert H.admit_clip(float(c), {"clip_coef": float(c)}) == float(c)
    assert H.admit_clip(float(c), None) == float(c)
    with pytest.raises(AssertionError):
        H.admit_clip(float(c), {"clip_coef": float(np.nextafter(up, np.float32(1)))})
