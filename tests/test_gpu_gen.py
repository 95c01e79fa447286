"""The CUDA twin of the input generator writes the same bits as the host version
(so full-size device inputs are the inputs the oracle sees)."""
import numpy as np
import pytest

import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    gen.build_cuda()
    return t


@pytest.mark.parametrize("dtype,sigma,scale", [(gen.FP16, 1e-3, 65536.0), (gen.FP16, 1e-3, 1.0),
                                               (gen.BF16, 1e-2, 1.0), (gen.FP16, 1.0, 3e4)])
def test_ranks_16_bitwise(torch, dtype, sigma, scale):
    nd, n, rs = 5, 100_003, 100_032
    d = torch.empty((nd, rs), dtype=torch.int16, device="cuda")
    gen.cuda_ranks_16(d.data_ptr(), 0, gen.STREAM_GRAD, 7, nd, n, sigma, scale, dtype,
                      rank_stride=rs, index0=12345)
    torch.cuda.synchronize()
    host = gen.ranks_16(0, gen.STREAM_GRAD, 7, nd, n, sigma, scale, dtype, rank_stride=rs,
                        index0=12345)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), host)


def test_f32_and_s16_bitwise(torch):
    n = 1_000_001
    d = torch.empty(n, dtype=torch.float32, device="cuda")
    gen.cuda_f32(d.data_ptr(), 3, gen.STREAM_MASTER, 0, 0, n, 0.02, index0=1 << 33)
    h = gen.f32(3, gen.STREAM_MASTER, 0, 0, n, 0.02, index0=1 << 33)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy().view(np.uint32), h.view(np.uint32))
    s = torch.empty(n, dtype=torch.int16, device="cuda")
    gen.cuda_s16(s.data_ptr(), 3, gen.STREAM_SHARD, 0, 9, n, 0.02, 1.0, gen.BF16)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint16),
                          gen.s16(3, gen.STREAM_SHARD, 0, 9, n, 0.02, 1.0, gen.BF16))
