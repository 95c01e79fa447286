"""The C-ABI library without a GPU: it builds, loads, exports every entry point
include/zero_b200.h declares, its host-only ledger functions agree with the
oracle, and invalid plans are rejected before anything touches CUDA."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zero_b200.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc needed to build")


@pytest.fixture(scope="module")
def z():
    from zero_sharded_mixed_02_gb300 import build
    build.build()
    import zero_sharded_mixed_02_gb300 as z
    z.lib()
    return z


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(
        r"^(?:zero_status_t|uint64_t|const char\*|int)\s+(zero_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for required in ("zero_plan_create", "zero_step", "zero_step_result", "zero_gather_layer",
                     "zero_state_bytes", "zero_comm_volume", "zero_plan_layout",
                     "zero_plan_destroy", "zero_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(z):
    L = ctypes.CDLL(z.LIB_PATH)
    for name in declared_entry_points():
        assert hasattr(L, name), name
    assert sorted(z.ENTRY_POINTS) == declared_entry_points()


def test_state_bytes_matches_oracle(z, oracle):
    for psi in (0, 1, 13, 1000, 7_500_000_000, 13_000_000_000, 10 ** 12):
        for nd in (1, 2, 3, 8, 16, 64, 1024):
            for stage in range(4):
                for K in (12, 16):
                    want = oracle.state_bytes(psi, nd, stage, K)
                    got = z.zero_state_bytes(psi, nd, stage, K)
                    # the library rounds the per-rank share up to whole bytes
                    assert want <= got < want + 1 + 1e-6 * want, (psi, nd, stage, K)


def test_comm_volume_and_capacity_match_oracle(z, oracle):
    for psi in (1, 1000, 7_500_000_000):
        for nd in (1, 4, 64):
            for stage in range(4):
                assert z.zero_comm_volume(psi, nd, stage, 0) == oracle.comm_volume(psi, nd, stage)
                w = oracle.comm_volume(psi, nd, stage, exact=1)
                assert w <= z.zero_comm_volume(psi, nd, stage, 1) < w + 1
    for mem in (32 * 10 ** 9, 80 * 10 ** 9):
        for nd in (1, 64, 256, 1024):
            for stage in range(4):
                want = oracle.max_params(mem, nd, stage)
                assert abs(z.zero_max_params(mem, nd, stage) - want) <= 1


def test_ledger_pages_examples(z):
    # the pages' worked examples, through the C ABI
    assert [z.zero_state_bytes(10 ** 9, 8, s) for s in range(4)] == [
        16 * 10 ** 9, 55 * 10 ** 8, 375 * 10 ** 7, 2 * 10 ** 9]
    assert [z.zero_state_bytes(75 * 10 ** 8, 64, s) for s in range(4)] == [
        120 * 10 ** 9, 31_406_250_000, 16_640_625_000, 1_875_000_000]
    assert z.zero_state_bytes(8 * 10 ** 9, 1, 0, K=16) == 160 * 10 ** 9
    assert z.zero_max_params(80 * 10 ** 9, 256, 3) == 1_280_000_000_000
    assert z.zero_comm_volume(10 ** 6, 4, 3, 1) == 2_250_000


def test_status_strings(z):
    assert z.zero_status_string(0) == "ZERO_OK"
    assert "invalid" in z.zero_status_string(1)


HP = None


@pytest.mark.parametrize("case", [
    dict(psi=10, nd=0), dict(psi=10, nd=2000), dict(psi=10, stage=4), dict(psi=10, stage=-1),
    dict(psi=11), dict(psi=10, dtype=7), dict(psi=10, hp=dict(loss_scale=0.0)),
    dict(psi=10, hp=dict(beta1=1.0)), dict(psi=10, hp=dict(eps=-1.0)),
    dict(psi=10, hp=dict(clip_norm=-1.0)), dict(psi=10, hp=dict(lr=float("nan"))),
    dict(psi=10, dtype=1, hp=dict(dynamic_scale=1)),
    dict(psi=10, hp=dict(dynamic_scale=1, backoff=0.0)),
])
def test_invalid_plans_rejected_before_cuda(z, case):
    shapes = [(2, 3), (4,)]
    hp = z.hparams(**case.get("hp", {}))
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan_create(case["psi"], case.get("nd", 2), case.get("stage", 1),
                           case.get("dtype", 0), shapes, hp)
    assert e.value.code == z.ZERO_EINVAL


@pytest.mark.parametrize("stage", [1, 3])
def test_psi_beyond_the_limit_rejected(z, stage):
    # 2^48 + 1 parameters in two tensors: the sizes add up, the plan is refused
    # before any device call
    shapes = [(1 << 24, 1 << 24), (1,)]
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan_create((1 << 48) + 1, 4, stage, 1, shapes, z.hparams())
    assert e.value.code == z.ZERO_EINVAL


def test_stage3_units_must_be_contiguous(z):
    shapes = [(4,), (4,), (4,)]
    with pytest.raises(z.ZeroError) as e:
        z.zero_plan_create(12, 2, 3, 1, shapes, z.hparams(), units=[0, 1, 0])
    assert e.value.code == z.ZERO_EINVAL


def test_null_plan_rejected(z):
    assert z.lib().zero_step(None, None, None, None, None, None, None, None) == z.ZERO_EINVAL
    assert z.lib().zero_step_result(None, None, None, None, None, None) == z.ZERO_EINVAL
    assert z.lib().zero_gather_layer(None, 0, None, None, None) == z.ZERO_EINVAL
    assert z.lib().zero_plan_destroy(None) == z.ZERO_OK
