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


@pytest.mark.parametrize("bits", [8, 4])
def test_quantized_unit_gather_bitwise(env, bits):
    torch, z = env
    w = W.scaled_llama(2, 256, 512, 8, 2, 1000, 16, W.llama3_8b())
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
