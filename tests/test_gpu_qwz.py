"""ZeRO++ quantized weight gather (qwZ) on the GPU against the oracle: the
block codes and scales bit for bit, and the dequantized unit gather bit for bit.
Every input is seeded (no oracle input comes from the GPU)."""
import numpy as np
import pytest

import gen
import oracle
from gen import workloads as W

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


def dev_codes(torch, n, bits):
    nbytes = n if bits == 8 else (n + 1) // 2
    return (torch.zeros(max(16, nbytes), dtype=torch.uint8, device="cuda"),
            torch.zeros(max(1, -(-n // 256)), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("n", [1, 7, 255, 256, 257, 1000, 65536 + 13, (1 << 20) + 3])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [gen.FP16, gen.BF16])
def test_quantize_shard_bitwise(env, n, bits, dtype):
    torch, z = env
    rng = np.random.default_rng(n)
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 1, n)).astype(np.float32)
    x[rng.integers(0, n, max(1, n // 5000))] *= 20           # a few outliers
    if n > 300:
        x[256:512] = 0.0                                       # an all-zero block
    x16 = oracle.from_float(dtype, x)
    d = torch.from_numpy(x16.view(np.int16)).cuda()
    codes, scales = dev_codes(torch, n, bits)
    z.zero_quantize_shard(dtype, d, n, bits, codes, scales, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    q, s = oracle.quantize_16(dtype, x16, bits, 256)
    assert np.array_equal(scales.cpu().numpy()[:s.size].view(np.uint32), s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy()[:q.size], q)


def _quantize_on_gpu(torch, z, dtype, x16, bits):
    n = x16.size
    d = torch.from_numpy(x16.view(np.int16)).cuda()
    codes, scales = dev_codes(torch, n, bits)
    z.zero_quantize_shard(dtype, d, n, bits, codes, scales,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [gen.FP16, gen.BF16])
def test_quantize_exact_ties_round_to_even(env, bits, dtype):
    """Blocks whose scale is a power of two and whose values are odd multiples of
    half that scale: every quotient is an exact tie k + 1/2, which must go to the
    even integer.  Values one 16-bit step either side of a tie are mixed in."""
    torch, z = env
    qmax = 127 if bits == 8 else 7
    rng = np.random.default_rng(100 + bits + dtype)
    nblk = 48
    x = np.empty(nblk * 256, np.float32)
    for b in range(nblk):
        scale = 2.0 ** (b % 20 - 10)
        k = rng.integers(-qmax, qmax, 256)                    # k + 1/2 in [-qmax + 1/2, qmax - 1/2]
        blk = (k + 0.5) * scale
        blk[rng.integers(0, 256)] = qmax * scale * (1 if b % 2 else -1)   # sets max|x|
        x[b * 256:(b + 1) * 256] = blk
    x16 = oracle.from_float(dtype, x)
    assert np.array_equal(oracle.to_float(dtype, x16), x)     # every value exact in 16 bits
    step = np.where(rng.random(x16.size) < 0.1, rng.choice([-1, 1], x16.size), 0)
    amax_pos = np.abs(x) == np.repeat(np.abs(x.reshape(nblk, 256)).max(1), 256)
    x16 = np.where(amax_pos, x16, (x16.astype(np.int32) + step).astype(np.uint16))
    q, s = oracle.quantize_16(dtype, x16, bits, 256)
    got_q, got_s = _quantize_on_gpu(torch, z, dtype, x16, bits)
    assert np.array_equal(got_s[:s.size].view(np.uint32), s.view(np.uint32))
    assert np.array_equal(got_q[:q.size], q)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [gen.FP16, gen.BF16])
def test_quantize_where_reciprocal_rounding_would_differ(env, bits, dtype):
    """A 4M-element input that, as checked here on the CPU, holds elements whose
    code from rounding x * fl(1/scale) differs from the code of the correctly
    rounded quotient x / scale: the GPU must still give the quotient's codes."""
    torch, z = env
    n = (1 << 22) + 77
    rng = np.random.default_rng(11 + bits + 3 * dtype)
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 1, n)).astype(np.float32)
    x16 = oracle.from_float(dtype, x)
    q, s = oracle.quantize_16(dtype, x16, bits, 256)
    xf = oracle.to_float(dtype, x16).astype(np.float32)
    sc = np.repeat(s, 256)[:n]
    live = sc != 0
    with np.errstate(all="ignore"):
        t = xf * (np.float32(1) / sc)
        y = xf / sc
    qmax = 127 if bits == 8 else 7
    differ = (np.clip(np.rint(t), -qmax, qmax) != np.clip(np.rint(y), -qmax, qmax)) & live
    assert np.count_nonzero(differ) >= 10
    got_q, got_s = _quantize_on_gpu(torch, z, dtype, x16, bits)
    assert np.array_equal(got_s[:s.size].view(np.uint32), s.view(np.uint32))
    assert np.array_equal(got_q[:q.size], q)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("dtype", [gen.FP16, gen.BF16])
def test_quantize_weight_like_blocks_near_half_integers(env, bits, dtype):
    """Weights like the ZeRO-3 workload's (16-bit N(0, 0.02)): with short
    mantissas, x / scale lands within 2^-14 of a half-integer for about one
    element in 300 (bf16) or 2500 (fp16), as counted here on the CPU; each of
    those codes must still be the correctly rounded quotient's."""
    torch, z = env
    n = (1 << 21) + 40
    x16 = gen.s16(5, gen.STREAM_SHARD, 0, 1, n, 0.02, 1.0, dtype)
    q, s = oracle.quantize_16(dtype, x16, bits, 256)
    xf = oracle.to_float(dtype, x16).astype(np.float32)
    sc = np.repeat(s, 256)[:n]
    with np.errstate(all="ignore"):
        y = xf / sc
    near = np.abs(np.abs(y - np.trunc(y)) - 0.5) < 2.0 ** -14
    assert np.count_nonzero(near) >= (2000 if dtype == gen.BF16 else 200)
    got_q, got_s = _quantize_on_gpu(torch, z, dtype, x16, bits)
    assert np.array_equal(got_s[:s.size].view(np.uint32), s.view(np.uint32))
    assert np.array_equal(got_q[:q.size], q)


def _ragged_units():
    """Units whose lengths leave every rank's slice, and the last rank's valid
    part, off any multiple of 8; several CTAs per slice."""
    import dataclasses
    return dataclasses.replace(W.llama3_8b(), name="ragged",
                               shapes=[(100003,), (70,), (4095, 1001), (13,), (2,)],
                               units=[0, 0, 1, 2, 2], nd=5)


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("model", ["llama-L2h256", "ragged"])
def test_quantized_unit_gather_bitwise(env, bits, model):
    torch, z = env
    w = (W.scaled_llama(2, 256, 512, 8, 2, 1000, 16, W.llama3_8b()) if model == "llama-L2h256"
         else _ragged_units())
    hp = z.hparams()
    plan = z.zero_plan_create(w.psi, w.nd, 3, w.dtype, w.shapes, hp, units=w.units)
    try:
        _, total, nunits, _ = z.zero_plan_layout(plan)
        sp = torch.cuda.current_stream().cuda_stream
        host_q, host_s, dev_q, dev_s = [], [], [], []
        for k in range(w.nd):
            x16 = gen.s16(7, gen.STREAM_SHARD, 0, k, total, 0.02, 1.0, w.dtype)
            q, s = oracle.quantize_16(w.dtype, x16, bits, 256)
            host_q.append(q)
            host_s.append(s)
            c, sc = dev_codes(torch, total, bits)
            z.zero_quantize_shard(w.dtype, torch.from_numpy(x16.view(np.int16)).cuda(), total,
                                  bits, c, sc, sp)
            dev_q.append(c)
            dev_s.append(sc)
        for u in range(nunits):
            ln, sl, off = z.zero_plan_unit(plan, u)
            out = torch.full((ln + 8,), -1, dtype=torch.int16, device="cuda")
            z.zero_gather_layer_q(plan, u, bits, dev_q, dev_s, out, sp)
            torch.cuda.synchronize()
            got = out.cpu().numpy().view(np.uint16)
            want = oracle.gather_unit_q(w.dtype, w.nd, ln, sl, off, bits, 256, host_q, host_s)
            assert np.array_equal(got[:ln], want)
            assert np.all(got[ln:] == 0xFFFF)
            # and close to the unquantized gather: relative L2 error of the block code
            plain = oracle.gather_unit(w.nd, ln, sl, [gen.s16(7, gen.STREAM_SHARD, 0, k, total, 0.02,
                                                              1.0, w.dtype)[off:off + sl]
                                                      for k in range(w.nd)])
            a = oracle.to_float(w.dtype, plain).astype(np.float64)
            b = oracle.to_float(w.dtype, got[:ln]).astype(np.float64)
            assert np.linalg.norm(a - b) / np.linalg.norm(a) < (0.01 if bits == 8 else 0.15)
    finally:
        z.zero_plan_destroy(plan)


def test_qwz_rejects_bad_arguments(env):
    torch, z = env
    x = torch.zeros(64, dtype=torch.int16, device="cuda")
    c, s = dev_codes(torch, 64, 8)
    for bits in (2, 16):
        with pytest.raises(z.ZeroError):
            z.zero_quantize_shard(1, x, 64, bits, c, s)
    with pytest.raises(z.ZeroError):
        z.zero_quantize_shard(1, x.data_ptr() + 2, 32, 8, c, s)
    plan = z.zero_plan_create(64, 4, 2, 1, [(64,)], z.hparams())
    try:
        with pytest.raises(z.ZeroError):                      # not a ZeRO-3 plan
            z.zero_gather_layer_q(plan, 0, 8, [c] * 4, [s] * 4, x)
    finally:
        z.zero_plan_destroy(plan)
