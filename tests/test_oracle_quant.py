"""Pins of the oracle's ZeRO++ block quantization (qwZ): the error figures the
lecture page prints, the round-to-nearest error bound, exact round trips, the
4-bit packing, and the quantized unit gather."""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "qwz_error.txt")


def _pins():
    out = []
    for line in open(GOLDEN, encoding="utf-8"):
        if not line.strip() or line.startswith("#"):
            continue
        body = line.split("|", 1)[0].split()
        out.append(pytest.param(int(body[0]), body[1], float(body[2]), float(body[3]),
                                id=f"int{body[0]}-{body[1]}"))
    return out


def _weights(seed, n=1_000_000):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(n).astype(np.float32)
    x[rng.choice(n, 64, replace=False)] *= 20.0
    return x


@pytest.mark.parametrize("bits,block,expected,tol", _pins())
def test_page_error_figures(oracle, bits, block, expected, tol):
    errs = []
    for seed in range(4):
        x = _weights(seed)
        b = x.size if block == "tensor" else int(block)
        q, s = oracle.quantize_f32(x, bits, b)
        y = oracle.dequantize_f32(q, s, x.size, bits, b)
        errs.append(100 * np.linalg.norm((x - y).astype(np.float64)) / np.linalg.norm(x.astype(np.float64)))
    assert abs(np.mean(errs) - expected) <= tol, errs


@pytest.mark.parametrize("bits", [8, 4])
def test_round_to_nearest_error_bound(oracle, bits):
    rng = np.random.default_rng(bits)
    x = (rng.standard_normal(100_003) * 10.0 ** rng.uniform(-3, 3, 100_003)).astype(np.float32)
    q, s = oracle.quantize_f32(x, bits, 256)
    y = oracle.dequantize_f32(q, s, x.size, bits, 256)
    scale = np.repeat(s, 256)[:x.size].astype(np.float64)
    assert np.all(np.abs(x.astype(np.float64) - y) <= scale * (0.5 + 1e-6))
    # the largest magnitude of each block maps to +-qmax
    qmax = 2 ** (bits - 1) - 1
    for b in range(0, x.size, 256):
        blk = x[b:b + 256]
        i = b + int(np.argmax(np.abs(blk)))
        assert abs(y[i]) == pytest.approx(qmax * s[b // 256], rel=1e-6)


@pytest.mark.parametrize("bits", [8, 4])
def test_exact_round_trip_on_the_grid(oracle, bits):
    # values that are integer multiples of a power-of-two scale, with the block
    # maximum at qmax: the scale is exact and the codes reproduce them exactly
    qmax = 2 ** (bits - 1) - 1
    rng = np.random.default_rng(7)
    k = rng.integers(-qmax, qmax + 1, (50, 256))
    k[:, 0] = qmax
    s = 2.0 ** rng.integers(-20, 5, (50, 1))
    x = (k * s).astype(np.float32).ravel()
    q, sc = oracle.quantize_f32(x, bits, 256)
    assert np.array_equal(sc, s.ravel().astype(np.float32))
    assert np.array_equal(oracle.dequantize_f32(q, sc, x.size, bits, 256), x)


def test_zero_block_and_int4_packing(oracle):
    q, s = oracle.quantize_f32(np.zeros(300, np.float32), 8, 256)
    assert not q.any() and not s.any()
    # absmax 7 -> scale 1 -> codes 1, -1, 7, -7; nibbles 1, F, 7, 9, low nibble first
    q, s = oracle.quantize_f32(np.array([1, -1, 7, -7], np.float32), 4, 256)
    assert s[0] == 1.0 and list(q) == [0xF1, 0x97]
    q, s = oracle.quantize_f32(np.array([1, -1, 127, -127], np.float32), 8, 256)
    assert list(q.view(np.int8)) == [1, -1, 127, -127]
    # round half to even: 0.5 and 1.5 and 2.5 at scale 1
    q, s = oracle.quantize_f32(np.array([0.5, 1.5, 2.5, -2.5, 127.0], np.float32), 8, 256)
    assert s[0] == 1.0 and list(q.view(np.int8)) == [0, 2, 2, -2, 127]


@pytest.mark.parametrize("dtype", [0, 1])
def test_quantized_unit_gather_is_dequantized_concatenation(oracle, dtype):
    rng = np.random.default_rng(dtype)
    nd, total, length, slice_, offset = 4, 4096, 3000, 768, 1024
    shards, qs, ss = [], [], []
    for _ in range(nd):
        x = (rng.standard_normal(total) * 0.02).astype(np.float32)
        x16 = oracle.from_float(dtype, x)
        q, s = oracle.quantize_16(dtype, x16, 8, 256)
        shards.append(oracle.dequantize_16(dtype, q, s, total, 8, 256))
        qs.append(q)
        ss.append(s)
    got = oracle.gather_unit_q(dtype, nd, length, slice_, offset, 8, 256, qs, ss)
    want = oracle.gather_unit(nd, length, slice_, [sh[offset:offset + slice_] for sh in shards])
    assert np.array_equal(got, want)
