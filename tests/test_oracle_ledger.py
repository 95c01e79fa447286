"""Pins of the oracle's memory ledger, capacity bound, communication volume and
flat partition against the numbers the pages print (tests/golden/ledger_pins.txt)."""
import math
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ledger_pins.txt")


def _pins():
    out = []
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        body, cite = line.split("|", 1)
        kind, psi, nd, stage, K, expected, tol = body.split()
        out.append(pytest.param(kind, float(psi), float(nd), int(stage), float(K),
                                float(expected), float(tol), id=f"{kind}-{psi}-{nd}-{stage}-K{K}"))
    return out


@pytest.mark.parametrize("kind,psi,nd,stage,K,expected,tol", _pins())
def test_ledger_pin(oracle, kind, psi, nd, stage, K, expected, tol):
    if kind == "state":
        got = oracle.state_bytes(psi, nd, stage, K)
    elif kind == "maxp":
        got = oracle.max_params(psi, nd, stage, K)
    elif kind == "comm":
        got = oracle.comm_volume(psi, nd, stage, exact=0)
    elif kind == "commx":
        got = oracle.comm_volume(psi, nd, stage, exact=1)
    elif kind == "ratio":
        got = oracle.state_bytes(1.0, nd, 0, K) / oracle.state_bytes(1.0, nd, stage, K)
    else:
        raise AssertionError(kind)
    if tol == 0:
        assert got == pytest.approx(expected, rel=1e-12, abs=0)
    else:
        assert abs(got - expected) <= tol * abs(expected), (got, expected)


def test_ledger_stage_order(oracle):
    # each stage removes one more redundancy: DP >= Z1 >= Z2 >= Z3 for any Nd >= 1,
    # with equality at Nd = 1 for Z3 (one rank holds everything)
    for psi in (1e6, 7.5e9):
        for nd in (1, 2, 8, 64, 1024):
            s = [oracle.state_bytes(psi, nd, st) for st in range(4)]
            assert s[0] >= s[1] >= s[2] >= s[3]
            if nd == 1:
                assert s[3] == s[0]


def test_comm_volume_is_allreduce_split(oracle):
    # an all-reduce is a reduce-scatter plus an all-gather (L18 3.1; PZ 7.1):
    # ZeRO-1/2 move exactly what DP moves; ZeRO-3 moves 1.5x
    for nd in (2, 4, 16, 64):
        dp = oracle.comm_volume(1e9, nd, 0, exact=1)
        assert oracle.comm_volume(1e9, nd, 1, exact=1) == dp
        assert oracle.comm_volume(1e9, nd, 2, exact=1) == dp
        assert oracle.comm_volume(1e9, nd, 3, exact=1) == pytest.approx(1.5 * dp)


def test_flat_partition_exercise(oracle):
    # L18 8. 练习 6 (参考答案): tensors of 100, 60 and 40 elements on 2 ranks; the
    # flat partition gives each rank 100 elements.  The oracle's shard length is
    # ceil(psi / nd) rounded to a multiple of 64 for the GPU layout; before that
    # rounding it is the page's 100.
    psi, nd = 100 + 60 + 40, 2
    assert math.ceil(psi / nd) == 100
    assert oracle.shard_elems(psi, nd) == 128            # 100 rounded up to 64s
    assert oracle.shard_elems(psi, nd) * nd >= psi


@pytest.mark.parametrize("psi,nd", [(1, 1), (5, 4), (13, 3), (16, 16), (1050112, 4),
                                    (124439808, 8), (1557611200, 16), (218112000, 64)])
def test_shard_layout_covers(oracle, psi, nd):
    s = oracle.shard_elems(psi, nd)
    assert s % 64 == 0
    assert s * nd >= psi                   # every element has an owner
    assert (s - 64) * nd < psi or s == 64  # no whole 64-block of slack per rank
