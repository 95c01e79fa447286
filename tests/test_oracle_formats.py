"""Pins of the oracle's 16-bit conversions against library routines (numpy
float16, torch bfloat16) and against the tie-to-even rule on exact midpoints."""
import numpy as np
import pytest
import torch

FP16, BF16 = 0, 1


def _bits32(x):
    return np.ascontiguousarray(x, np.float32).view(np.uint32)


def _edge_floats():
    """float32 values around every interesting boundary of both formats."""
    rng = np.random.default_rng(0)
    vals = [0.0, -0.0, np.inf, -np.inf, np.nan,
            65504.0, 65519.996, 65520.0, 65520.004, 65535.0, 65536.0, 1e30,
            2.0 ** -14, 2.0 ** -15, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26,
            np.finfo(np.float32).max, np.finfo(np.float32).tiny, 1e-45, 3.3895314e38,
            3.3961776e38, 1.0 + 2 ** -8, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11]
    x = np.array(vals, np.float32)
    rnd_bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    rnd = rnd_bits.view(np.float32)
    near = (rng.standard_normal(500_000) * 10.0 ** rng.integers(-9, 5, 500_000)).astype(np.float32)
    return np.concatenate([x, -x, rnd, near])


def test_half_to_float_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.to_float(FP16, bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(_bits32(ours[~nan]), _bits32(ref[~nan]))   # signed zeros too


def test_bf16_to_float_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.to_float(BF16, bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(_bits32(ours[~nan]), _bits32(ref[~nan]))


def test_float_to_half_matches_numpy(oracle):
    x = _edge_floats()
    ours = oracle.from_float(FP16, x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(np.isnan(ours[nan].view(np.float16)))


def test_float_to_bf16_matches_torch(oracle):
    x = _edge_floats()
    ours = oracle.from_float(BF16, x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_roundtrip_every_finite_pattern(oracle, dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.to_float(dtype, bits)
    keep = np.isfinite(f)
    back = oracle.from_float(dtype, f[keep])
    assert np.array_equal(back, bits[keep])


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_midpoints_round_to_even(oracle, dtype):
    # every midpoint between two adjacent positive finite values (and between the
    # largest finite value and the first value past it) is exact in binary32 and
    # must round to the neighbour whose last fraction bit is 0
    lo_bits = np.arange(0, 0x7C00 if dtype == FP16 else 0x7F80, dtype=np.uint32).astype(np.uint16)
    hi_bits = (lo_bits.astype(np.uint32) + 1).astype(np.uint16)
    lo = oracle.to_float(dtype, lo_bits).astype(np.float64)
    if dtype == FP16:
        hi = np.where(hi_bits == 0x7C00, 65536.0, oracle.to_float(dtype, hi_bits).astype(np.float64))
    else:
        hi = np.where(hi_bits == 0x7F80, 2.0 ** 128,
                      oracle.to_float(dtype, hi_bits).astype(np.float64))
    mid64 = (lo + hi) / 2
    mid = mid64.astype(np.float32)
    exact = mid.astype(np.float64) == mid64
    assert exact.all()
    got = oracle.from_float(dtype, mid)
    want = np.where(lo_bits % 2 == 0, lo_bits, hi_bits)
    assert np.array_equal(got, want)
    got_neg = oracle.from_float(dtype, -mid)
    assert np.array_equal(got_neg, want | 0x8000)
