"""Pins of the oracle's shard regrouping (sharded checkpoint restored at another
rank count or stage).

[Z026] sec. 5 (restoring a sharded checkpoint at another degree of parallelism
must regroup ownership, keep the parameter order and keep each element's
moments together).  The regrouping is pinned against the unit split and gather
(themselves pinned to numpy's concatenation), closed forms for rank counts that
divide one another, round trips and a padding check.
"""
import numpy as np
import pytest


def shard_by_units(oracle, nd, lens, flat):
    """Rank shards of the 16-bit vector `flat` built from the pinned unit split:
    rank r's shard is the concatenation of its slice of every unit."""
    per_rank = [[] for _ in range(nd)]
    start = 0
    for n in lens:
        sl = oracle.shard_unit(nd, flat[start:start + n], oracle.shard_elems(n, nd))
        for r in range(nd):
            per_rank[r].append(sl[r])
        start += n
    return [np.concatenate(p) for p in per_rank]


def gather_by_units(oracle, nd, lens, shards):
    """The flat vector back from rank shards through the pinned unit gather."""
    out, off = [], 0
    for n in lens:
        s = oracle.shard_elems(n, nd)
        out.append(oracle.gather_unit(nd, n, s, [sh[off:off + s] for sh in shards]))
        off += s
    return np.concatenate(out) if out else np.zeros(0, np.uint16)


LAYOUTS = [
    (4, [1000]),                       # stages 0-2: one unit
    (3, [300_001]),
    (16, [64 * 16 * 5]),               # divides exactly, no padding
    (5, [7, 130, 4096, 1, 999]),       # stage 3: several units, ragged slices
    (8, [64, 64, 640, 77]),
    (1, [10, 20]),
]


@pytest.mark.parametrize("nd,lens", LAYOUTS)
def test_layout_shard_len_and_global(oracle, nd, lens):
    L = oracle.Layout(nd, lens)
    assert L.shard_len() == sum(oracle.shard_elems(n, nd) for n in lens)
    seen = np.zeros(L.psi, np.int64)
    for r in range(nd):
        for j in range(L.shard_len()):
            g = L.global_index(r, j)
            if g >= 0:
                seen[g] += 1
    assert np.all(seen == 1)                          # every flat index held exactly once
    assert L.global_index(0, L.shard_len()) == -1     # past the shard: nothing


@pytest.mark.parametrize("a", LAYOUTS)
@pytest.mark.parametrize("b_nd", [1, 2, 7, 16])
def test_reshard_matches_unit_split_and_gather(oracle, a, b_nd):
    nd, lens = a
    psi = sum(lens)
    rng = np.random.default_rng(psi + b_nd)
    flat = rng.integers(0, 65536, psi).astype(np.uint16)
    A = oracle.Layout(nd, lens)
    old = shard_by_units(oracle, nd, lens, flat)
    assert np.array_equal(gather_by_units(oracle, nd, lens, old), flat)
    for b_lens in ([psi], lens):                       # to stages 0-2, and to stage 3 units
        B = oracle.Layout(b_nd, b_lens)
        new = oracle.reshard(A, old, B)
        want = shard_by_units(oracle, b_nd, b_lens, flat)
        for r in range(b_nd):
            assert np.array_equal(new[r], want[r]), (r, b_lens)


def test_reshard_to_one_rank_is_the_concatenation(oracle):
    """Stages 0-2: the flat vector is the concatenation of the shards, trimmed."""
    psi, nd = 100_003, 6
    A = oracle.Layout(nd, [psi])
    S = A.shard_len()
    rng = np.random.default_rng(1)
    old = [rng.standard_normal(S).astype(np.float32) for _ in range(nd)]
    new = oracle.reshard(A, old, oracle.Layout(1, [psi]))
    cat = np.concatenate(old)
    assert np.array_equal(new[0][:psi].view(np.uint32), cat[:psi].view(np.uint32))
    assert not new[0][psi:].any()


def test_reshard_halving_rank_count_joins_pairs(oracle):
    """psi = 8 * 4096: Nd 8 -> 4 gives rank r the shards 2r and 2r+1 joined;
    Nd 8 -> 16 splits each shard in two."""
    psi = 8 * 4096
    A = oracle.Layout(8, [psi])
    old = [np.arange(r * 4096, (r + 1) * 4096, dtype=np.uint32) * 3 + 1 for r in range(8)]
    four = oracle.reshard(A, old, oracle.Layout(4, [psi]))
    for r in range(4):
        assert np.array_equal(four[r], np.concatenate([old[2 * r], old[2 * r + 1]]))
    sixteen = oracle.reshard(A, old, oracle.Layout(16, [psi]))
    for r in range(16):
        assert np.array_equal(sixteen[r], old[r // 2][(r % 2) * 2048:(r % 2 + 1) * 2048])


@pytest.mark.parametrize("a,b", [((4, [1000]), (3, [1000])), ((5, [7, 130, 4096, 1, 999]),
                                                                 (2, [5233])),
                                 ((8, [64, 64, 640, 77]), (3, [128, 717]))])
def test_reshard_round_trip_and_padding(oracle, a, b):
    A, B = oracle.Layout(*a), oracle.Layout(*b)
    rng = np.random.default_rng(7)
    old = [rng.integers(1, 2**32 - 1, A.shard_len(), dtype=np.uint64).astype(np.uint32)
           for _ in range(A.nd)]                     # padding holds nonzero garbage
    mid = oracle.reshard(A, old, B)
    back = oracle.reshard(B, mid, A)
    for r in range(A.nd):
        valid = np.array([A.global_index(r, j) >= 0 for j in range(A.shard_len())])
        assert np.array_equal(back[r][valid], old[r][valid])
        assert not back[r][~valid].any()               # padding comes back as zero
    for r in range(B.nd):
        valid = np.array([B.global_index(r, j) >= 0 for j in range(B.shard_len())])
        assert not mid[r][~valid].any() and np.all(mid[r][valid] != 0)
