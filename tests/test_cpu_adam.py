"""The library's host Adam (ZeRO-Offload, [L18] sec. 4.4) against the oracle, on the
CPU: it needs no GPU.

- its 16-bit conversions, exhaustively for binary16 / bfloat16 -> binary32 and
  on every kind of binary32 value (ties, subnormals, overflow, NaN) the other
  way (with beta1 = 0 and lr = 0 the update reduces to m = g, p unchanged);
- the update, bit for bit against the oracle's Adam on the oracle's unscaled
  gradient, for both 16-bit types, the three weight-decay modes, clipping,
  ragged sizes and several thread counts.
"""
import numpy as np
import pytest

import oracle as _oracle_mod

FP16, BF16 = 0, 1


@pytest.fixture(scope="module")
def z():
    from zero_sharded_mixed_02_gb300 import build
    build.build()
    import zero_sharded_mixed_02_gb300 as zz
    zz.lib()
    return zz


def run_cpu(z, g16, dtype, S, c, bc1, bc2, hp, master, m, v, nthreads=0):
    master, m, v = master.copy(), m.copy(), v.copy()
    params = np.full(master.size, 0xA5A5, np.uint16)
    z.zero_cpu_adam(g16, dtype, master.size, S, c, bc1, bc2, hp, master, m, v, params, nthreads)
    return master, m, v, params


def same_or_both_nan(a, b):
    return np.all((a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b)))


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_widening_every_16_bit_code(z, oracle, dtype):
    codes = np.arange(65536, dtype=np.uint16)
    n = codes.size
    hp = z.hparams(lr=0.0, beta1=0.0, beta2=0.5, eps=1.0)
    master = np.zeros(n, np.float32)
    _, m, _, _ = run_cpu(z, codes, dtype, 1.0, 1.0, 1.0, 1.0, hp, master, master, master)
    # m = 0 * m + 1 * g: the sum turns -0 into +0, so compare with +0 + g
    with np.errstate(invalid="ignore"):
        want = np.float32(0.0) + oracle.to_float(dtype, codes)
    assert same_or_both_nan(m, want)


def special_floats(rng):
    vals = [
        np.array([0.0, -0.0, np.inf, -np.inf, np.nan, -np.nan, 65504.0, 65519.99, 65520.0,
                  65536.0, 1e30, -1e30, 5.96e-8, 2.98e-8, 2.9802322e-08, 1e-45, -1e-45,
                  6.1035156e-05, 6.1e-05, 3.4028235e38, 1.0, -1.0], np.float32),
        rng.standard_normal(200_000).astype(np.float32) * np.float32(10.0) **
        rng.integers(-9, 6, 200_000).astype(np.float32),
        # exact midpoints between neighbouring binary16 values (every normal binade)
        ((np.arange(1, 0x7BFF, dtype=np.uint32).astype(np.uint16).view(np.float16)
          .astype(np.float64) + np.arange(2, 0x7C00, dtype=np.uint32).astype(np.uint16)
          .view(np.float16).astype(np.float64)) / 2).astype(np.float32),
        # and between neighbouring bfloat16 values
        (((np.arange(0x0080, 0x7F7F, 7, dtype=np.uint32) << 16) | 0x8000).view(np.float32)),
        rng.integers(0, 2**32, 500_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    return np.concatenate(vals)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_narrowing_ties_subnormals_overflow_nan(z, oracle, dtype):
    rng = np.random.default_rng(dtype)
    x = special_floats(rng)
    hp = z.hparams(lr=0.0, beta1=0.0, beta2=0.5, eps=1.0)
    g16 = np.zeros(x.size, np.uint16)
    zero = np.zeros(x.size, np.float32)
    master, _, _, params = run_cpu(z, g16, dtype, 1.0, 1.0, 1.0, 1.0, hp, x, zero, zero)
    assert same_or_both_nan(master, x)                 # lr = 0: p unchanged
    want = oracle.from_float(dtype, x)
    nan = np.isnan(x)
    assert np.array_equal(params[~nan], want[~nan])
    assert np.array_equal(params[nan], want[nan])     # quiet NaN, sign kept, like the oracle


CASES = [
    dict(dtype=FP16, S=65536.0, c=0.37, wd=0.0, decoupled=1, t=1),
    dict(dtype=FP16, S=1024.0, c=1.0, wd=0.01, decoupled=1, t=7),
    dict(dtype=BF16, S=1.0, c=0.5, wd=0.1, decoupled=0, t=3),
    dict(dtype=BF16, S=3.0, c=1.0, wd=0.0, decoupled=1, t=1000),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"dt{c['dtype']}-wd{c['wd']}-d{c['decoupled']}")
@pytest.mark.parametrize("n", [1, 63, 64, 65, 1000, 1_000_003])
def test_update_matches_the_oracle(z, oracle, case, n):
    rng = np.random.default_rng(n)
    dtype, S = case["dtype"], case["S"]
    raw = (rng.standard_normal(n) * 0.05 * S).astype(np.float32)
    g16 = oracle.from_float(dtype, raw)
    master = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32)
    opt = _oracle_mod.Opt(lr=1e-3, weight_decay=case["wd"], decoupled_wd=case["decoupled"])
    hp = z.hparams(lr=1e-3, weight_decay=case["wd"], decoupled_wd=case["decoupled"])
    b1t, b2t = 1.0, 1.0
    for _ in range(case["t"]):                      # beta^t by repeated double products
        b1t *= float(np.float32(0.9))
        b2t *= float(np.float32(0.999))
    bc1, bc2 = np.float32(1.0 - b1t), np.float32(1.0 - b2t)
    _, g, _ = oracle.reduce16(1, dtype, g16[None, :], loss_scale=S)   # the oracle's unscaled g
    want = [master.copy(), m.copy(), v.copy(), np.zeros(n, np.uint16)]
    oracle.adam(g, np.float32(case["c"]), *want, dtype, opt, float(bc1), float(bc2))
    for threads in (1, 3, 0):
        got = run_cpu(z, g16, dtype, S, case["c"], float(bc1), float(bc2), hp, master, m, v,
                      threads)
        for k, (a, b) in enumerate(zip(got, want)):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (k, threads)


def test_argument_checks(z):
    hp = z.hparams()
    x = np.zeros(4, np.float32)
    p = np.zeros(4, np.uint16)
    for args in ((None, 0, 4, 1.0, 1.0, 1.0, 1.0, hp, x, x, x, p),
                 (p, 2, 4, 1.0, 1.0, 1.0, 1.0, hp, x, x, x, p),
                 (p, 0, 4, 0.0, 1.0, 1.0, 1.0, hp, x, x, x, p),
                 (p, 0, 4, 1.0, 1.0, 0.0, 1.0, hp, x, x, x, p),
                 (p, 0, 4, 1.0, 1.0, 1.0, 1.0, hp, x, None, x, p)):
        with pytest.raises(z.ZeroError) as e:
            z.zero_cpu_adam(*args)
        assert e.value.code == z.ZERO_EINVAL
    z.zero_cpu_adam(p, 0, 0, 1.0, 1.0, 1.0, 1.0, hp, x, x, x, p)      # n = 0: nothing to do
