"""The seeded input generator (host side) and the workload shape lists."""
import numpy as np
import pytest
import torch

import gen
from gen import workloads


def test_splitmix64_published_sequence():
    # SplitMix64 seeded with 0 starts 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4,
    # 0x06c45d188009454f (Steele, Lea & Flood's generator)
    assert [gen.mix(k * gen.GOLDEN) for k in (1, 2, 3)] == [
        0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_key_matches_python_statement():
    for args in [(0, 1, 0, 0), (0, 1, 7, 15), (123456789, 3, 2, 63), (2 ** 63 + 5, 2, 0, 1)]:
        assert gen.host().zgen_key(*args) == gen.key(*args)


@pytest.mark.parametrize("dtype", [gen.FP16, gen.BF16])
def test_16bit_inputs_are_library_rounding_of_f32(dtype):
    # the 16-bit inputs are the nearest-even rounding of the binary32 sample
    v = gen.f32(0, gen.STREAM_GRAD, 3, 5, 200_000, 1e-3, scale=65536.0)
    b = gen.s16(0, gen.STREAM_GRAD, 3, 5, 200_000, 1e-3, scale=65536.0, dtype=dtype)
    if dtype == gen.FP16:
        ref = v.astype(np.float16).view(np.uint16)
    else:
        ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)


def test_moments_and_bounds():
    sigma = 0.02
    v = gen.f32(0, gen.STREAM_MASTER, 0, 0, 1_000_000, sigma).astype(np.float64)
    assert abs(v.mean()) < 3 * sigma / 1000
    assert v.std() == pytest.approx(sigma, rel=0.01)
    assert np.abs(v).max() <= 3.4642 * sigma


def test_rank_layout_and_padding():
    a = gen.ranks_16(0, gen.STREAM_GRAD, 1, 3, 100, 1e-2, 1.0, gen.BF16, rank_stride=128)
    assert a.shape == (3, 128) and not a[:, 100:].any()
    for r in range(3):
        assert np.array_equal(a[r, :100],
                              gen.s16(0, gen.STREAM_GRAD, 1, r, 100, 1e-2, 1.0, gen.BF16))
    assert not np.array_equal(a[0, :100], a[1, :100])
    # an index offset continues the same sequence
    tail = gen.s16(0, gen.STREAM_GRAD, 1, 2, 40, 1e-2, 1.0, gen.BF16, index0=60)
    assert np.array_equal(tail, a[2, 60:100])
    idx = np.array([99, 0, 17])
    assert np.array_equal(gen.s16_at(0, gen.STREAM_GRAD, 1, 1, idx, 1e-2, 1.0, gen.BF16),
                          a[1, idx])


def test_inf_site_in_range():
    for step in (3, 7):
        r, i = gen.inf_site(0, step, 1557611200, 16)
        assert 0 <= r < 16 and 0 <= i < 1557611200
    assert gen.inf_site(0, 3, 10**9, 16) != gen.inf_site(0, 7, 10**9, 16)


def test_workload_parameter_counts():
    # counts of the shape lists: tiny (4 tensors), GPT-2 small (148), GPT-2 1.5B
    # (580), LLaMA-3-8B (291 tensors, 34 ZeRO-3 units)
    assert workloads.tiny().psi == 512 * 1024 + 1024 + 1024 * 512 + 512 == 1050112
    g2 = workloads.gpt2_small()
    assert (g2.psi, len(g2.shapes)) == (124439808, 148)
    xl = workloads.gpt2_xl()
    assert (xl.psi, len(xl.shapes)) == (1557611200, 580)
    ll = workloads.llama3_8b()
    assert (ll.psi, len(ll.shapes), len(ll.unit_lengths())) == (8030261248, 291, 34)
    assert ll.unit_lengths()[1] == 218112000
