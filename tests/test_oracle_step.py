"""Pins of the oracle's optimizer step.

Nothing here re-types the oracle's loops: each test checks a consequence that
the pages or the mathematics fix -- the fixed rank order of the reduce, exact
averages, closed forms of Adam at step 1 and under a constant gradient, the
scale invariance of Adam, decoupled decay under a zero gradient, the clipped
norm, the overflow skip with its loss-scale schedule, and the invariant that a
sharded step equals the unsharded one bit for bit.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

FP16, BF16 = 0, 1


def f16(x):
    """numpy (library) rounding of float values to fp16 bit patterns."""
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def bf16(x):
    """torch (library) rounding of float values to bf16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits16(dtype, x):
    return f16(x) if dtype == FP16 else bf16(x)


def val16(dtype, b):
    b = np.asarray(b, np.uint16)
    if dtype == FP16:
        return b.view(np.float16).astype(np.float64)
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(x).astype(np.float64)


def state(n, seed=0):
    rng = np.random.default_rng(seed)
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    return master, np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)


# --------------------------------------------------------------------- reduce
def test_reduce_left_fold_in_rank_order(oracle):
    # L18 2.5: the emulated collectives sum in a fixed rank order.  With ranks
    # (65504, -65504, 2^-24) the fold 0 + r0 + r1 + r2 keeps the tiny term;
    # the reverse order loses it to rounding.
    grads = f16(np.array([[65504.0], [-65504.0], [2.0 ** -24]]))
    g, ovf = oracle.reduce(3, FP16, grads)
    assert not ovf
    assert g[0] == np.float32(2.0 ** -24) / np.float32(3)
    g_rev, _ = oracle.reduce(3, FP16, grads[::-1].copy())
    assert g_rev[0] == 0.0


@pytest.mark.parametrize("nd", [1, 2, 3, 4, 5, 8, 16])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_reduce_identical_ranks_is_identity(oracle, nd, dtype):
    # every rank holds the same gradient: its average is that gradient exactly
    # (k*x is exact in binary32 for k <= 16 and 16-bit x; (k x)/k = x)
    rng = np.random.default_rng(nd)
    x = bits16(dtype, rng.standard_normal(777) * 10.0 ** rng.integers(-6, 3, 777))
    grads = np.tile(x, (nd, 1))
    g, ovf = oracle.reduce(nd, dtype, grads)
    assert not ovf
    assert np.array_equal(g, val16(dtype, x).astype(np.float32))


@pytest.mark.parametrize("nd", [2, 4, 8, 16])
def test_reduce_exact_average_and_unscale(oracle, nd):
    # small-integer multiples of 2^-6 sum exactly; the average over a power-of-two
    # nd and the unscale by a power-of-two loss scale are exact scalings
    rng = np.random.default_rng(nd)
    ints = rng.integers(-500, 500, size=(nd, 1000))
    grads = f16(ints * 2.0 ** -6)
    for scale in (1.0, 1024.0, 65536.0):
        g, _ = oracle.reduce(nd, FP16, grads, loss_scale=scale)
        want = [float(Fraction(int(s), 64 * nd) / Fraction(scale)) for s in ints.sum(0)]
        assert np.array_equal(g.astype(np.float64), np.array(want))


def test_reduce_nd1_is_the_cast(oracle):
    rng = np.random.default_rng(1)
    x = f16(rng.standard_normal(4096) * 100)
    g, _ = oracle.reduce(1, FP16, x[None, :], loss_scale=1024.0)
    assert np.array_equal(g, (x.view(np.float16).astype(np.float32) / np.float32(1024)))


def test_reduce_overflow_flag(oracle):
    base = f16(np.ones((4, 10)))
    assert oracle.reduce(4, FP16, base)[1] is False
    for bad in (np.inf, -np.inf, np.nan):
        g = base.copy()
        g[2, 7] = f16([bad])[0]
        assert oracle.reduce(4, FP16, g)[1] is True
    big = f16(np.full((16, 3), 65504.0))            # 16 x max half is finite in fp32
    assert oracle.reduce(16, FP16, big)[1] is False


# ----------------------------------------------------------------------- norm
def test_norm_matches_numpy(oracle):
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(100_003) * 1e-3).astype(np.float32)
    ref = np.linalg.norm(g.astype(np.float64))
    assert math.sqrt(oracle.sumsq(g)) == pytest.approx(ref, rel=1e-13)
    assert oracle.sumsq(np.zeros(0, np.float32)) == 0.0


def test_clip_coefficient(oracle):
    assert oracle.clip_coef(10.0, 1.0) == np.float32(0.1)
    assert oracle.clip_coef(0.5, 1.0) == 1.0
    assert oracle.clip_coef(1.0, 1.0) == 1.0          # clip only when above
    assert oracle.clip_coef(1e9, 0.0) == 1.0          # 0 = off


# --------------------------------------------------------- Adam closed forms
def _run(oracle, nd, dtype, grads_list, opt, master, m, v, params, scale=1.0, **kw):
    st = oracle.new_scalars(scale)
    res = []
    for grads in grads_list:
        res.append(oracle.step(nd, dtype, grads, master, m, v, params, opt, st, **kw))
    return st, res


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_adam_step1_closed_form(oracle, dtype):
    # At t = 1 with m = v = 0 and bias correction, m_hat = g and v_hat = g^2, so
    # the update is -lr g / (|g| + eps).  Magnitudes near eps check where eps goes.
    n, nd = 4000, 4
    rng = np.random.default_rng(5)
    mags = 10.0 ** rng.uniform(-9 if dtype == BF16 else -4, 1, n)
    x = bits16(dtype, rng.choice([-1.0, 1.0], n) * mags)
    g = val16(dtype, x)
    master, m, v, params = state(n)
    p0 = master.astype(np.float64).copy()
    opt = oracle.Opt(lr=1e-3, eps=1e-8)
    _run(oracle, nd, dtype, [np.tile(x, (nd, 1))], opt, master, m, v, params)
    want = p0 - 1e-3 * g / (np.abs(g) + np.float64(np.float32(1e-8)))
    err = np.abs(master.astype(np.float64) - want)
    assert np.all(err <= 2 * ulp32(want) + 1e-3 * 4e-7)
    assert np.array_equal(params, bits16(dtype, master))   # stage 5 cast of the master


def test_adam_constant_gradient_closed_form(oracle):
    # With the same gradient every step, m_hat_t = g and v_hat_t = g^2 for all t
    # (bias correction removes the (1 - beta^t) factors), so after T steps the
    # master has moved by -T lr g / (|g| + eps).
    n, nd, T = 3000, 8, 12
    rng = np.random.default_rng(6)
    x = bf16(rng.standard_normal(n) * 10.0 ** rng.uniform(-5, 0, n))
    g = val16(BF16, x)
    master, m, v, params = state(n, seed=1)
    p0 = master.astype(np.float64).copy()
    opt = oracle.Opt(lr=1e-3)
    st, res = _run(oracle, nd, BF16, [np.tile(x, (nd, 1))] * T, opt, master, m, v, params)
    assert st.t == T and all(r["skipped"] == 0 for r in res)
    want = p0 - T * 1e-3 * g / (np.abs(g) + np.float64(np.float32(1e-8)))
    err = np.abs(master.astype(np.float64) - want)
    assert np.all(err <= T * (ulp32(want) + 1e-3 * 4e-6))
    # the bias corrections it used were 1 - beta^T
    assert res[-1]["bc1"] == np.float32(1 - np.float64(np.float32(0.9)) ** T)
    assert res[-1]["bc2"] == np.float32(1 - np.float64(np.float32(0.999)) ** T)


def test_adam_scale_invariance_eps0(oracle):
    # With eps = 0, scaling every gradient by 2^k scales m by 2^k and v by 4^k
    # exactly and leaves the master bit-identical.
    n, nd = 2000, 4
    rng = np.random.default_rng(7)
    # scale the rounded fp16 values (exact), not the values before rounding
    seq = [val16(FP16, f16(rng.standard_normal((nd, n)) * 0.01)) for _ in range(4)]
    out = []
    for k in (0, 5):
        master, m, v, params = state(n, seed=2)
        _run(oracle, nd, FP16, [f16(s * 2.0 ** k) for s in seq], oracle.Opt(eps=0.0),
             master, m, v, params)
        out.append((master, m, v))
    (p0, m0, v0), (p5, m5, v5) = out
    assert np.array_equal(p0, p5)
    assert np.array_equal(m0 * np.float32(32), m5)
    assert np.array_equal(v0 * np.float32(1024), v5)


def test_adamw_zero_gradient_decay(oracle):
    # zero gradient: m = v = 0 and the Adam term is 0 / eps = 0, so decoupled
    # decay alone moves the master: p_T = p_0 (1 - lr wd)^T
    n, nd, T = 1000, 2, 7
    master, m, v, params = state(n, seed=3)
    p0 = master.astype(np.float64).copy()
    opt = oracle.Opt(lr=1e-3, weight_decay=0.01, decoupled_wd=1)
    _run(oracle, nd, BF16, [np.zeros((nd, n), np.uint16)] * T, opt, master, m, v, params)
    want = p0 * (1 - np.float64(np.float32(1e-3)) * np.float64(np.float32(0.01))) ** T
    assert np.all(np.abs(master - want) <= T * ulp32(want))
    assert not m.any() and not v.any()


def test_adam_l2_decay_step1(oracle):
    # coupled (L2) decay with a zero gradient: g_eff = wd p, and at t = 1 the
    # update is -lr g_eff / (|g_eff| + eps)
    n, nd = 1000, 2
    master, m, v, params = state(n, seed=4)
    p0 = master.astype(np.float64).copy()
    opt = oracle.Opt(lr=1e-3, weight_decay=0.01, decoupled_wd=0)
    _run(oracle, nd, BF16, [np.zeros((nd, n), np.uint16)], opt, master, m, v, params)
    ge = np.float64(np.float32(0.01)) * p0
    want = p0 - 1e-3 * ge / (np.abs(ge) + np.float64(np.float32(1e-8)))
    assert np.all(np.abs(master - want) <= 2 * ulp32(want) + 1e-3 * 4e-7)


def test_clip_scales_gradient_to_threshold(oracle):
    # clip by global norm: the clipped gradient has norm exactly the threshold, and
    # at t = 1 the first moment is (1 - beta1) times the clipped gradient
    n, nd = 5000, 4
    rng = np.random.default_rng(8)
    grads = bf16(rng.standard_normal((nd, n)) * 0.05)
    g_avg, _ = oracle.reduce(nd, BF16, grads)
    norm = np.linalg.norm(g_avg.astype(np.float64))
    assert norm > 1.0
    master, m, v, params = state(n)
    _, (res,) = _run(oracle, nd, BF16, [grads], oracle.Opt(clip_norm=1.0), master, m, v, params)
    assert res["grad_norm"] == pytest.approx(norm, rel=1e-13)
    assert res["clip_coef"] == np.float32(1.0 / norm)
    clipped = m.astype(np.float64) / np.float64(np.float32(1 - np.float64(np.float32(0.9))))
    assert np.linalg.norm(clipped) == pytest.approx(1.0, rel=1e-6)
    # below the threshold nothing is scaled
    master, m, v, params = state(n)
    _, (res,) = _run(oracle, nd, BF16, [grads], oracle.Opt(clip_norm=1e6), master, m, v, params)
    assert res["clip_coef"] == 1.0


# ---------------------------------------------------- overflow and loss scale
def test_overflow_skips_step_and_halves_scale(oracle):
    n, nd = 600, 4
    rng = np.random.default_rng(9)
    opt = oracle.Opt(dynamic_scale=1, backoff=0.5, growth_interval=2)
    master, m, v, params = state(n)
    st = oracle.new_scalars(1024.0)
    good = f16(rng.standard_normal((nd, n)) * 1e-3 * 1024)
    oracle.step(nd, FP16, good, master, m, v, params, opt, st)
    assert (st.t, st.loss_scale, st.good_steps) == (1, 1024.0, 1)
    snap = [a.copy() for a in (master, m, v, params)]
    bad = good.copy()
    bad[3, 17] = f16([np.inf])[0]
    r = oracle.step(nd, FP16, bad, master, m, v, params, opt, st)
    assert r["skipped"] == 1 and r["overflow"] == 1
    assert (st.t, st.loss_scale, st.good_steps) == (1, 512.0, 0)
    for a, b in zip(snap, (master, m, v, params)):
        assert np.array_equal(a, b)                          # state bit-unchanged
    # two good steps in a row double the scale (growth_interval = 2)
    for k in range(2):
        r = oracle.step(nd, FP16, good, master, m, v, params, opt, st)
        assert r["skipped"] == 0
    assert (st.t, st.loss_scale, st.good_steps) == (3, 1024.0, 0)
    # a NaN also skips
    bad[0, 0] = f16([np.nan])[0]
    assert oracle.step(nd, FP16, bad, master, m, v, params, opt, st)["skipped"] == 1


def test_static_scale_reports_overflow_without_skipping(oracle):
    n, nd = 64, 2
    master, m, v, params = state(n)
    st = oracle.new_scalars(8.0)
    grads = f16(np.ones((nd, n)))
    grads[1, 5] = f16([np.inf])[0]
    r = oracle.step(nd, FP16, grads, master, m, v, params, oracle.Opt(dynamic_scale=0), st)
    assert r["overflow"] == 1 and r["skipped"] == 0 and st.t == 1 and st.loss_scale == 8.0


def _warm_state(oracle, nd, n, dtype, opt, seed):
    """state after one ordinary step, so m and v are nonzero"""
    rng = np.random.default_rng(seed)
    master, m, v, params = state(n, seed)
    st = oracle.new_scalars(1.0)
    oracle.step(nd, dtype, bits16(dtype, rng.standard_normal((nd, n)) * 0.03), master, m, v,
                params, opt, st)
    return [master, m, v, params], st, rng


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_static_scale_overflow_without_clip_touches_only_its_element(oracle, dtype):
    """With a static scale and no clip nothing global gates the update: the
    non-finite element's state becomes non-finite, and every other element is
    updated bit for bit as if that element's gradient had been finite."""
    n, nd, site = 300, 4, (2, 77)
    opt = oracle.Opt(dynamic_scale=0)
    s0, st0, rng = _warm_state(oracle, nd, n, dtype, opt, 11)
    grads = bits16(dtype, rng.standard_normal((nd, n)) * 0.03)
    bad = grads.copy()
    bad[site] = bits16(dtype, [np.inf])[0]
    fine = grads.copy()
    fine[site] = 0
    a = [x.copy() for x in s0]
    b = [x.copy() for x in s0]
    sa, sb = oracle.new_scalars(1.0), oracle.new_scalars(1.0)
    for sx in (sa, sb):
        sx.t, sx.beta1_pow, sx.beta2_pow = st0.t, st0.beta1_pow, st0.beta2_pow
    ra = oracle.step(nd, dtype, bad, *a, opt, sa)
    rb = oracle.step(nd, dtype, fine, *b, opt, sb)
    assert ra["overflow"] == 1 and ra["skipped"] == 0 and rb["overflow"] == 0
    assert sa.t == sb.t == 2
    assert not np.isfinite(ra["grad_norm"]) and ra["clip_coef"] == 1.0
    keep = np.arange(n) != site[1]
    for x, y in zip(a, b):
        assert np.array_equal(x[keep], y[keep])
    # g = +inf: m and v become +inf, the update inf/inf = NaN reaches the master
    assert np.isposinf(a[1][site[1]]) and np.isposinf(a[2][site[1]]) and np.isnan(a[0][site[1]])


def test_static_scale_overflow_with_clip_is_a_zero_gradient_step(oracle):
    """With a static scale and clipping, a non-finite gradient makes the norm
    infinite and the clip coefficient tau / inf = 0: every finite element takes
    exactly the step a zero gradient gives (m *= beta1, v *= beta2, the master
    moves by the remaining momentum), and the non-finite element becomes NaN
    (inf * 0)."""
    n, nd, site = 256, 3, (0, 200)
    opt = oracle.Opt(dynamic_scale=0, clip_norm=1.0)
    s0, st0, rng = _warm_state(oracle, nd, n, BF16, opt, 12)
    assert np.count_nonzero(s0[1]) == n
    bad = bf16(rng.standard_normal((nd, n)) * 0.03)
    bad[site] = bf16([np.inf])[0]
    zero = np.zeros((nd, n), np.uint16)
    a = [x.copy() for x in s0]
    b = [x.copy() for x in s0]
    sa, sb = oracle.new_scalars(1.0), oracle.new_scalars(1.0)
    for sx in (sa, sb):
        sx.t, sx.beta1_pow, sx.beta2_pow = st0.t, st0.beta1_pow, st0.beta2_pow
    ra = oracle.step(nd, BF16, bad, *a, opt, sa)
    rb = oracle.step(nd, BF16, zero, *b, opt, sb)
    assert ra["overflow"] == 1 and ra["skipped"] == 0 and ra["clip_coef"] == 0.0
    assert rb["grad_norm"] == 0.0 and rb["clip_coef"] == 1.0
    keep = np.arange(n) != site[1]
    for x, y in zip(a, b):
        assert np.array_equal(x[keep], y[keep])
    b1 = np.float32(0.9)
    assert np.array_equal(a[1][keep], (b1 * s0[1][keep]).astype(np.float32))   # m *= beta1
    assert np.isnan(a[0][site[1]]) and np.isnan(a[1][site[1]]) and np.isnan(a[2][site[1]])


@pytest.mark.parametrize("clip", [0.0, 1.0])
def test_skip_on_overflow_under_a_static_scale(oracle, clip):
    """skip_on_overflow = 1 with a static scale: an overflow skips the step
    (state bit-unchanged, t unchanged) and the scale is not backed off; the
    next clean step proceeds as step t + 1."""
    n, nd = 200, 4
    opt = oracle.Opt(dynamic_scale=0, skip_on_overflow=1, clip_norm=clip)
    s0, st, rng = _warm_state(oracle, nd, n, FP16, opt, 13)
    st.loss_scale = 4.0
    snap = [x.copy() for x in s0]
    bad = f16(rng.standard_normal((nd, n)) * 0.03 * 4.0)
    bad[1, 3] = f16([np.nan])[0]
    r = oracle.step(nd, FP16, bad, *s0, opt, st)
    assert r["overflow"] == 1 and r["skipped"] == 1
    assert (st.t, st.loss_scale, st.good_steps) == (1, 4.0, 0)
    for x, y in zip(snap, s0):
        assert np.array_equal(x, y)
    good = f16(rng.standard_normal((nd, n)) * 0.03 * 4.0)
    r = oracle.step(nd, FP16, good, *s0, opt, st)
    assert r["skipped"] == 0 and st.t == 2 and st.loss_scale == 4.0
    # without skip_on_overflow the same overflow is reported and not skipped
    r = oracle.step(nd, FP16, bad, *s0, oracle.Opt(dynamic_scale=0, clip_norm=clip), st)
    assert r["overflow"] == 1 and r["skipped"] == 0 and st.t == 3 and st.loss_scale == 4.0


# ------------------------------------------ sharded == unsharded (L18 2.5)
def _seq(rng, nd, n, steps, dtype):
    return [bits16(dtype, rng.standard_normal((nd, n)) * 10.0 ** rng.uniform(-4, 0))
            for _ in range(steps)]


@pytest.mark.parametrize("n", [1, 5, 13, 16, 1000, 4099])
@pytest.mark.parametrize("nd", [1, 2, 3, 4, 8, 16])
def test_sharded_equals_unsharded(oracle, n, nd):
    rng = np.random.default_rng(n * 100 + nd)
    dtype = FP16 if (n + nd) % 2 else BF16
    seq = _seq(rng, nd, n, 3, dtype)
    opt = oracle.Opt(weight_decay=0.01, dynamic_scale=int(dtype == FP16))
    ref = state(n)
    st_ref = oracle.new_scalars(1.0)
    for gr in seq:
        r_ref = oracle.step(nd, dtype, gr, *ref, opt, st_ref)
    smin = -(-n // nd)
    for shard in sorted({smin, oracle.shard_elems(n, nd), n}):
        for nthreads in (1, 3):
            got = state(n)
            st = oracle.new_scalars(1.0)
            for gr in seq:
                r = oracle.step_sharded(nd, dtype, gr, *got, opt, st, shard=shard,
                                        nthreads=nthreads)
            for a, b in zip(ref, got):
                assert np.array_equal(a, b)
            assert r["grad_norm"] == pytest.approx(r_ref["grad_norm"], rel=1e-14)
            assert (st.t, st.loss_scale) == (st_ref.t, st_ref.loss_scale)


def test_every_shard_assignment_tiny(oracle):
    # Psi <= 8: every equal contiguous split gives the same result (clip off)
    for n in range(1, 9):
        for nd in (1, 2, 3, 4, 8):
            rng = np.random.default_rng(n * 10 + nd)
            seq = _seq(rng, nd, n, 2, BF16)
            ref = state(n)
            st_ref = oracle.new_scalars()
            for gr in seq:
                oracle.step(nd, BF16, gr, *ref, oracle.Opt(), st_ref)
            for shard in range(-(-n // nd), n + 1):
                got = state(n)
                st = oracle.new_scalars()
                for gr in seq:
                    oracle.step_sharded(nd, BF16, gr, *got, oracle.Opt(), st, shard=shard)
                for a, b in zip(ref, got):
                    assert np.array_equal(a, b)


def test_wrong_ownership_is_detectable(oracle):
    # Z026 三: a rank that updates its slice with only its own local gradient
    # (no reduce) changes the algorithm; the averaged-gradient step must differ.
    n, nd = 256, 4
    rng = np.random.default_rng(11)
    grads = f16(rng.standard_normal((nd, n)))
    a = state(n)
    oracle.step(nd, FP16, grads, *a, oracle.Opt(), oracle.new_scalars())
    b = state(n)
    local = np.tile(grads[0], (nd, 1))                 # rank 0's gradient everywhere
    oracle.step(nd, FP16, local, *b, oracle.Opt(), oracle.new_scalars())
    assert not np.array_equal(a[0], b[0])


# ------------------------------------------------------ ZeRO-3 unit gather
@pytest.mark.parametrize("nd,length", [(1, 1), (4, 5), (8, 4160), (64, 218112), (3, 1000)])
def test_gather_inverts_shard(oracle, nd, length):
    rng = np.random.default_rng(length)
    unit = rng.integers(0, 65536, length).astype(np.uint16)
    slice_elems = oracle.shard_elems(length, nd)
    slices = oracle.shard_unit(nd, unit, slice_elems)
    flat = np.concatenate(slices)
    assert np.array_equal(flat[:length], unit) and not flat[length:].any()
    assert np.array_equal(oracle.gather_unit(nd, length, slice_elems, slices), unit)


# ------------------------------------------- brute force against the textbook
def textbook_steps(nd, dtype, grads_per_step, master, S, clip, lr, wd, b1f, b2f, eps):
    """Mixed-precision Adam/AdamW steps of the pages' method written out in
    float64 (16-bit inputs exact in float64; every operation ~1e-16 relative),
    with the fp16 dynamic loss scale (skip and halve on overflow)."""
    p = master.astype(np.float64)
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    t, out = 0, []
    b1, b2 = float(b1f), float(b2f)
    for g16 in grads_per_step:
        x = np.stack([val16(dtype, g16[r]) for r in range(nd)])
        g = x.sum(axis=0) / nd / S
        if not np.all(np.isfinite(g)):
            S = S / 2
            out.append(("skip", S))
            continue
        norm = math.sqrt(float(np.sum(g * g)))
        c = clip / norm if clip > 0 and norm > clip else 1.0
        t += 1
        bc1, bc2 = 1.0 - b1 ** t, 1.0 - b2 ** t
        p = p * (1.0 - lr * wd)
        m = b1 * m + (1.0 - b1) * (g * c)
        v = b2 * v + (1.0 - b2) * (g * c) ** 2
        p = p - lr * (m / bc1) / (np.sqrt(v / bc2) + eps)
        out.append(("step", norm))
    return p, m, v, S, out


@pytest.mark.parametrize("n", [5, 13, 16])
@pytest.mark.parametrize("nd", [1, 2, 3, 4, 8, 16])
def test_brute_force_against_the_textbook(oracle, n, nd):
    """Tiny models, every rank count of the configurations: three steps (the
    second with an injected inf) of the oracle against the float64 textbook.
    The oracle rounds each binary32 operation, so the two agree to a few
    binary32 ulps on master, m, v and to 1 ulp on the 16-bit params."""
    rng = np.random.default_rng(100 * n + nd)
    S, clip, lr, wd = 1024.0, 0.05, 1e-3, 0.01
    steps = []
    for k in range(3):
        g = f16(rng.standard_normal((nd, n)) * 1e-2 * S)
        if k == 1:
            g[nd - 1, n // 2] = 0x7C00
        steps.append(g)
    master0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    opt = oracle.Opt(lr=lr, weight_decay=wd, decoupled_wd=1, clip_norm=clip, dynamic_scale=1)
    st = oracle.new_scalars(S)
    master, m, v, params = master0.copy(), *state(n)[1:]
    res = [oracle.step(nd, FP16, g, master, m, v, params, opt, st) for g in steps]
    tp, tm, tv, tS, tout = textbook_steps(nd, FP16, steps, master0, S, clip, lr, wd,
                                          np.float32(0.9), np.float32(0.999), np.float32(1e-8))
    assert [r["skipped"] for r in res] == [0, 1, 0] and [o[0] for o in tout] == ["step", "skip", "step"]
    assert st.loss_scale == tS == S / 2 and st.t == 2
    for r, o in zip(res, tout):
        if o[0] == "step":
            # each g is one binary32 rounding (or two: fold, divide) off the real value
            assert abs(r["grad_norm"] - o[1]) <= 1e-6 * o[1]
    # a few binary32 ulps: 1e-5 relative, plus 1e-6 of the array's largest value
    # where the update nearly cancels the old value (a dropped term or a wrong
    # sign is off by about lr = 1e-3 of the master's scale)
    for got, want in ((master, tp), (m, tm), (v, tv)):
        err = np.abs(got.astype(np.float64) - want)
        assert np.all(err <= 1e-5 * np.abs(want) + 1e-6 * np.abs(want).max()), err.max()
    keys = lambda b: np.where(b & 0x8000, -(b & 0x7FFF).astype(np.int32), (b & 0x7FFF).astype(np.int32))
    assert np.max(np.abs(keys(params) - keys(f16(tp)))) <= 1
