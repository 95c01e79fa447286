"""Pins of the oracle's ZeRO-Offload step ([L18] sec. 4.4; [ZL8] sec. 6.2, 7): the
averaged gradient crosses the link in the 16-bit type and the host unscales it.

Pinned by: the identity at Nd = 1, agreement with the (separately pinned)
unrounded reduce through numpy's / torch's own 16-bit rounding, hand-computed
ties to even, and exact agreement with the plain step whenever the rank mean
is representable in the 16-bit type.
"""
import numpy as np
import pytest

FP16, BF16 = 0, 1


def lib16(dtype, x32):
    """Library rounding of binary32 values to the 16-bit type (bits)."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == FP16:
        return x32.astype(np.float16).view(np.uint16)
    torch = pytest.importorskip("torch")
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def widen(dtype, b):
    if dtype == FP16:
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << 16).view(np.float32)      # bfloat16: the upper half


def grads16(dtype, rng, nd, n, scale=1.0):
    x = (rng.standard_normal((nd, n)) * scale).astype(np.float32)
    return lib16(dtype, x.ravel()).reshape(nd, n)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_one_rank_copies_the_gradient_unchanged(oracle, dtype):
    rng = np.random.default_rng(dtype)
    g = grads16(dtype, rng, 1, 50_000, 3.0)
    g16, gf, ovf = oracle.reduce16(1, dtype, g, loss_scale=1024.0)
    assert not ovf and np.array_equal(g16, g[0])
    want, _ = oracle.reduce(1, dtype, g, loss_scale=1024.0)
    assert np.array_equal(gf.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("nd", [2, 3, 5, 16])
def test_rounds_the_pinned_mean_to_16_bits(oracle, dtype, nd):
    """The copied value is the 16-bit rounding of the unrounded mean (the plain
    reduce times a power-of-two scale, exact), and the host divides it by S."""
    rng = np.random.default_rng(nd)
    S = 256.0
    g = grads16(dtype, rng, nd, 40_000, 4.0)
    g16, gf, ovf = oracle.reduce16(nd, dtype, g, loss_scale=S)
    plain, _ = oracle.reduce(nd, dtype, g, loss_scale=S)
    mean = plain * np.float32(S)
    assert not ovf
    assert np.array_equal(g16, lib16(dtype, mean))
    assert np.array_equal(gf.view(np.uint32), (widen(dtype, g16) / np.float32(S)).view(np.uint32))
    if nd in (3, 5):                                   # rounding does change some values
        assert not np.array_equal(gf, plain)


@pytest.mark.parametrize("dtype,pairs", [
    (FP16, [((0x3C00, 0x3C01), 0x3C00),        # 1 + 2^-11: halfway, to the even 1.0
            ((0x3C01, 0x3C02), 0x3C02),        # 1 + 3*2^-11: halfway, to the even neighbour
            ((0xBC01, 0xBC02), 0xBC02)]),      # the same, negative
    (BF16, [((0x3F80, 0x3F81), 0x3F80),        # 1 + 2^-8
            ((0x3F81, 0x3F82), 0x3F82),
            ((0xBF81, 0xBF82), 0xBF82)]),
])
def test_ties_go_to_even(oracle, dtype, pairs):
    for (a, b), want in pairs:
        g = np.array([[a], [b]], np.uint16)
        g16, _, _ = oracle.reduce16(2, dtype, g)
        assert int(g16[0]) == want, (hex(a), hex(b), hex(int(g16[0])))
    # not a tie: (1 + 1 + (1 + 2^-10)) / 3 = 1 + 2^-10/3 is nearer 1.0
    one, up = (0x3C00, 0x3C01) if dtype == FP16 else (0x3F80, 0x3F81)
    g16, _, _ = oracle.reduce16(3, dtype, np.array([[one], [one], [up]], np.uint16))
    assert int(g16[0]) == one


def run_both(oracle, nd, dtype, grads, opt, scale, steps=1):
    n = grads.shape[1]
    rng = np.random.default_rng(5)
    init = (rng.standard_normal(n) * 0.02).astype(np.float32)
    a = [init.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    b = [x.copy() for x in a]
    sa, sb = oracle.new_scalars(scale), oracle.new_scalars(scale)
    ra = [oracle.step(nd, dtype, grads, *a, opt, sa) for _ in range(steps)]
    rb = [oracle.step_offload(nd, dtype, grads, *b, opt, sb) for _ in range(steps)]
    return a, b, ra, rb, sa, sb


@pytest.mark.parametrize("nd", [3, 7, 16])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_equals_the_plain_step_when_the_mean_is_representable(oracle, nd, dtype):
    """Every rank holds the same gradient: the fp32 fold is nd * x exactly and
    the mean is x, so nothing is rounded and the two steps agree bit for bit."""
    rng = np.random.default_rng(nd + 10 * dtype)
    scale = 65536.0 if dtype == FP16 else 1.0
    row = grads16(dtype, rng, 1, 30_000, 0.05 * scale)[0]       # unscaled norm ~ 8.7
    grads = np.tile(row, (nd, 1))
    opt = oracle.Opt(clip_norm=1.0, dynamic_scale=1 if dtype == FP16 else 0, weight_decay=0.01)
    a, b, ra, rb, sa, sb = run_both(oracle, nd, dtype, grads, opt, scale, steps=2)
    assert ra == rb and ra[0]["skipped"] == 0 and ra[0]["clip_coef"] < 1.0
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    assert (sa.t, sa.loss_scale) == (sb.t, sb.loss_scale)


def test_step_composes_reduce16_norm_clip_and_adam(oracle):
    rng = np.random.default_rng(3)
    nd, n, S = 4, 20_000, 1024.0
    grads = grads16(FP16, rng, nd, n, 0.5 * S)
    opt = oracle.Opt(clip_norm=0.5)
    init = (rng.standard_normal(n) * 0.02).astype(np.float32)
    state = [init.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    st = oracle.new_scalars(S)
    res = oracle.step_offload(nd, FP16, grads, *state, opt, st)
    _, g, ovf = oracle.reduce16(nd, FP16, grads, loss_scale=S)
    norm = np.sqrt(oracle.sumsq(g))
    assert res["grad_norm"] == norm and not ovf
    c = oracle.clip_coef(norm, 0.5)
    assert res["clip_coef"] == c < 1.0
    want = [init.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.uint16)]
    r2 = oracle.advance(opt, oracle.new_scalars(S), ovf)
    oracle.adam(g, c, *want, FP16, opt, r2.bc1, r2.bc2)
    for x, y in zip(state, want):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_overflow_skips_under_dynamic_scaling(oracle):
    rng = np.random.default_rng(4)
    grads = grads16(FP16, rng, 4, 1000, 10.0)
    grads[2, 17] = 0x7C00                                 # +inf from one rank
    opt = oracle.Opt(dynamic_scale=1)
    init = np.ones(1000, np.float32)
    state = [init.copy(), np.zeros(1000, np.float32), np.zeros(1000, np.float32),
             np.zeros(1000, np.uint16)]
    st = oracle.new_scalars(4096.0)
    res = oracle.step_offload(4, FP16, grads, *state, opt, st)
    assert res["skipped"] == 1 and st.loss_scale == 2048.0 and st.t == 0
    assert np.array_equal(state[0], init) and not state[3].any()
