"""Sharded checkpoints on the GPU ([Z026] sec. 5; [L32] sec. 4.3).

- the files hold exactly the device state, in the documented format (read here
  by an independent reader that also recomputes every block checksum);
- save, then load into a fresh plan with the same layout, then step on: the
  same results as stepping on without the round trip;
- reshard: a checkpoint saved at Nd = 16 (stage 2) or by the ranks of a
  ZeRO-3 plan loads into plans of other rank counts and stages; the loaded
  state equals the oracle's state regrouped by the oracle (zo_reshard), and the
  steps that follow match the oracle continuing at the new rank count;
- failures: a missing rank file or manifest, a truncated or damaged file, a
  file from another step and another model are refused with explicit errors.
"""
import dataclasses
import os

import numpy as np
import pytest

import gen
import harness as H
import oracle

pytestmark = pytest.mark.gpu

BE = 1 << 20
GOLD = np.uint64(0x9E3779B97F4A7C15)


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


# ------------------------------------------- an independent reader of the format
def zck64(buf, w0):
    b = np.frombuffer(bytes(buf), np.uint8)
    if b.size % 8:
        b = np.concatenate([b, np.zeros(8 - b.size % 8, np.uint8)])
    x = b.view("<u8")
    with np.errstate(over="ignore"):
        zz = x + np.arange(w0 + 1, w0 + 1 + x.size, dtype=np.uint64) * GOLD
        zz = (zz ^ (zz >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        zz = (zz ^ (zz >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        zz = zz ^ (zz >> np.uint64(31))
        return int(zz.sum(dtype=np.uint64))


SCALARS = [("loss_scale", "<f4"), ("good_steps", "<i4"), ("t", "<i8"), ("b1", "<f8"), ("b2", "<f8")]
MANIFEST = np.dtype([("magic", "S8"), ("version", "<u4"), ("size", "<u4"), ("psi", "<u8"),
                     ("nd", "<i4"), ("stage", "<i4"), ("dtype", "<i4"), ("zero", "<i4"),
                     ("model_hash", "<u8")] + SCALARS + [("meta_hash", "<u8")])
SHARD = np.dtype([("magic", "S8"), ("version", "<u4"), ("header_bytes", "<u4"), ("psi", "<u8"),
                  ("nd", "<i4"), ("stage", "<i4"), ("dtype", "<i4"), ("rank", "<i4"),
                  ("model_hash", "<u8")] + SCALARS +
                 [("nseg", "<u8"), ("n", "<u8"), ("block_elems", "<u8"), ("nblocks", "<u8"),
                  ("table_offset", "<u8"), ("array_offset", "<u8", (4,)), ("file_bytes", "<u8"),
                  ("meta_hash", "<u8")])
assert MANIFEST.itemsize == 88 and SHARD.itemsize == 168


def read_manifest(d):
    raw = open(os.path.join(d, "manifest.zck"), "rb").read()
    assert len(raw) == 88
    m = np.frombuffer(raw, MANIFEST)[0]
    assert m["magic"] == b"ZEROMAN1" and int(m["meta_hash"]) == zck64(raw[:80], 0)
    return m


def read_shard(path):
    """Header, segments [(global_start, count)] and the four arrays; every block
    checksum and the header checksum recomputed."""
    raw = open(path, "rb").read()
    h = np.frombuffer(raw[:168], SHARD)[0]
    assert h["magic"] == b"ZEROSHD1" and int(h["version"]) == 1
    nseg, n, nb = int(h["nseg"]), int(h["n"]), int(h["nblocks"])
    assert int(h["block_elems"]) == BE and nb == -(-n // BE) and len(raw) == int(h["file_bytes"])
    t0 = int(h["table_offset"])
    table = np.frombuffer(raw[t0:t0 + 8 * (2 * nseg + 4 * nb)], "<u8")
    assert (zck64(raw[:160], 0) + zck64(table.tobytes(), 0)) % (1 << 64) == int(h["meta_hash"])
    segs = table[:2 * nseg].reshape(-1, 2).astype(np.int64)
    hashes = table[2 * nseg:].reshape(4, nb) if nb else np.zeros((4, 0), np.uint64)
    arrays = []
    for a, dt in enumerate(("<f4", "<f4", "<f4", "<u2")):
        es = 4 if a < 3 else 2
        off = int(h["array_offset"][a])
        assert off % 4096 == 0
        data = raw[off:off + n * es]
        for b in range(nb):
            blk = data[b * BE * es:min((b + 1) * BE, n) * es]
            assert zck64(blk, b * BE * es // 8) == int(hashes[a, b]), (path, a, b)
        arrays.append(np.frombuffer(data, dt))
    return h, segs, arrays


# ------------------------------------------------------------- layouts (test side)
def unit_lens(c):
    if c.stage <= 2:
        return [c.psi]
    sizes = [int(np.prod(s)) for s in c.shapes]
    units = c.units or list(range(len(sizes)))
    lens = [0] * (max(units) + 1)
    for u, n in zip(units, sizes):
        lens[u] += n
    return lens


def index_map(nd, lens, r):
    """Flat index held at each position of rank r's shard (-1: padding)."""
    parts, start = [], 0
    for n in lens:
        s = oracle.shard_elems(n, nd)
        loc = r * s + np.arange(s, dtype=np.int64)
        parts.append(np.where(loc < n, start + loc, -1))
        start += n
    return np.concatenate(parts) if parts else np.zeros(0, np.int64)


def test_index_map_agrees_with_the_oracle_layout():
    for nd, lens in ((16, [4_049_654]), (5, [3_000_001, 77, 1_048_576])):
        L = oracle.Layout(nd, lens)
        for r in (0, nd // 2, nd - 1):
            mp = index_map(nd, lens, r)
            assert mp.size == L.shard_len()
            for j in np.random.default_rng(r).integers(0, mp.size, 200):
                assert mp[j] == L.global_index(r, int(j))


# ------------------------------------------------------------------ GPU plumbing
class State:
    """A plan plus its device buffers (stages 0-2: the flat buffers; stage 3:
    the resident shard of one rank)."""

    def __init__(self, torch, z, c):
        self.torch, self.z, self.c = torch, z, c
        self.plan = z.zero_plan_create(c.psi, c.nd, c.stage, c.dtype, c.shapes, c.hparams(z),
                                       units=c.units if c.stage == 3 else None)
        shard, self.padded, _, ws = z.zero_plan_layout(self.plan)
        dev = torch.device("cuda", 0)
        self.master = torch.zeros(self.padded, dtype=torch.float32, device=dev)
        self.m = torch.zeros_like(self.master)
        self.v = torch.zeros_like(self.master)
        self.params = torch.zeros(self.padded, dtype=torch.int16, device=dev)
        self.work = torch.empty(max(ws, 16) // 4, dtype=torch.float32, device=dev) if ws else None
        self.grads = None

    def bufs(self):
        return self.master, self.m, self.v, self.params

    def fill(self, value):
        for b in (self.master, self.m, self.v):
            b.fill_(value)
        self.params.fill_(int(np.int16(np.uint16(0xBEEF).view(np.int16))))

    def host(self):
        self.torch.cuda.synchronize()
        return (self.master.cpu().numpy(), self.m.cpu().numpy(), self.v.cpu().numpy(),
                self.params.cpu().numpy().view(np.uint16))

    def step(self, g):
        """g: [nd][padded] 16-bit gradients (host)."""
        if self.grads is None:
            self.grads = self.torch.empty((self.c.nd, self.padded), dtype=self.torch.int16,
                                          device="cuda")
        self.grads.copy_(self.torch.from_numpy(np.ascontiguousarray(g).view(np.int16)))
        self.z.zero_step(self.plan, self.grads, *self.bufs(), self.work,
                         self.torch.cuda.current_stream().cuda_stream)
        r = self.z.zero_step_result(self.plan)
        r["overflow"] = self.z.zero_step_overflow(self.plan)
        return r

    def save(self, d, rank=-1, flags=0):
        self.z.zero_checkpoint_save(self.plan, str(d), rank, *self.bufs(), flags)

    def load(self, d, rank=-1):
        self.z.zero_checkpoint_load(self.plan, str(d), rank, *self.bufs())

    def close(self):
        self.z.zero_plan_destroy(self.plan)


def flat_init(c):
    return gen.f32(c.seed, gen.STREAM_MASTER, 0, 0, c.psi, 0.02)


def run_steps(st, c, steps, scale):
    """Steps (1-based numbers) on a stages 0-2 State; returns results and the scale."""
    out = []
    for k in steps:
        r = st.step(H.grads_for_step(c, k, c.psi, st.padded, scale))
        out.append(r)
        scale = r["loss_scale"]
    return out, scale


def oracle_steps(c, steps, state, st_scalars, follow=None):
    """The oracle's steps; follow: the GPU's results of the same steps, whose
    clip coefficients the oracle admits (harness.admit_clip)."""
    master, m, v, params = state
    res = []
    for i, k in enumerate(steps):
        g = np.ascontiguousarray(H.grads_for_step(c, k, c.psi, c.psi, st_scalars.loss_scale))
        r = H.oracle_step_admitting(c.nd, c.dtype, g, master, m, v, params, c.opt(), st_scalars,
                                    follow[i] if follow else None, what=f"step {k}")
        r["loss_scale"] = st_scalars.loss_scale
        r["t"] = st_scalars.t
        res.append(r)
    return res


def flat_of(c, host):
    return tuple(x[:c.psi] for x in host)


BASE = H.Case(shapes=[(3_000_001,), (77,), (1_048_576,)], nd=16, dtype=gen.FP16,
              grad_sigma=1e-3, loss_scale=65536.0, dynamic_scale=1, growth_interval=2,
              inf_steps=(2,), steps=3)


# ------------------------------------------------------------------ the files
@pytest.mark.parametrize("nd", [4, 16])
def test_files_hold_the_state(env, tmp_path, nd):
    torch, z = env
    c = dataclasses.replace(BASE, nd=nd)
    st = State(torch, z, c)
    try:
        st.master[:c.psi] = torch.from_numpy(flat_init(c)).cuda()
        res, _ = run_steps(st, c, (1, 2, 3), c.loss_scale)
        st.save(tmp_path)
        host = st.host()
        man = read_manifest(tmp_path)
        assert (int(man["psi"]), int(man["nd"]), int(man["stage"]), int(man["dtype"])) == \
            (c.psi, nd, 2, c.dtype)
        assert float(man["loss_scale"]) == res[-1]["loss_scale"] and int(man["t"]) == res[-1]["t"]
        S = oracle.shard_elems(c.psi, nd)
        names = sorted(os.listdir(tmp_path))
        assert names == ["manifest.zck"] + [f"shard_{r:05d}_of_{nd:05d}.zck" for r in range(nd)]
        for r in range(nd):
            h, segs, arrays = read_shard(tmp_path / f"shard_{r:05d}_of_{nd:05d}.zck")
            assert int(h["rank"]) == r and int(h["t"]) == res[-1]["t"]
            lo, hi = r * S, min((r + 1) * S, c.psi)
            assert segs.tolist() == ([[lo, hi - lo]] if hi > lo else [])
            for a in range(4):
                want = host[a][lo:hi]
                assert np.array_equal(arrays[a].view(want.dtype), want), (r, a)
    finally:
        st.close()


# -------------------------------------------------------- resume, same layout
def test_resume_continues_bit_for_bit(env, tmp_path):
    """Save after step 3, step twice; a fresh plan loading the checkpoint and
    taking the same two steps ends in the same state and reports."""
    torch, z = env
    c = BASE
    a = State(torch, z, c)
    b = State(torch, z, c)
    try:
        a.master[:c.psi] = torch.from_numpy(flat_init(c)).cuda()
        _, scale = run_steps(a, c, (1, 2, 3), c.loss_scale)
        a.save(tmp_path)
        ra, _ = run_steps(a, c, (4, 5), scale)
        b.fill(7.0)
        b.load(tmp_path)
        rb, _ = run_steps(b, c, (4, 5), z.zero_step_result(b.plan)["loss_scale"])
        for x, y in zip(ra, rb):
            assert x == y
        for x, y in zip(a.host(), b.host()):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
        # step 4 is the second good step since the skip: the scale grows only
        # because the good-step count was restored with the state
        assert ra[0]["loss_scale"] == 2 * 32768.0
    finally:
        a.close()
        b.close()


# ------------------------------------------------------------------ reshard
TARGETS = [dict(nd=8, stage=2), dict(nd=3, stage=1), dict(nd=1, stage=0),
           dict(nd=5, stage=3)]


def expected_shards(c_old, flat_state, c_new):
    """The oracle's flat state regrouped into c_new's layout by the oracle."""
    A = oracle.Layout(1, [c_old.psi])                 # the flat vector as one rank
    B = oracle.Layout(c_new.nd, unit_lens(c_new))
    out = []
    for x in flat_state:
        one = np.zeros(A.shard_len(), x.dtype)
        one[:c_old.psi] = x
        out.append(oracle.reshard(A, [one], B))
    return out


@pytest.mark.parametrize("target", TARGETS, ids=lambda t: f"nd{t['nd']}-stage{t['stage']}")
def test_reshard_matches_oracle_and_continues(env, tmp_path, target):
    torch, z = env
    c = BASE
    a = State(torch, z, c)
    try:
        a.master[:c.psi] = torch.from_numpy(flat_init(c)).cuda()
        ra, scale = run_steps(a, c, (1, 2, 3), c.loss_scale)
        a.save(tmp_path)
        saved = flat_of(c, a.host())
    finally:
        a.close()
    # the oracle's own three steps
    ostate = [flat_init(c), np.zeros(c.psi, np.float32), np.zeros(c.psi, np.float32),
              np.zeros(c.psi, np.uint16)]
    osc = oracle.new_scalars(c.loss_scale)
    ores = oracle_steps(c, (1, 2, 3), ostate, osc, follow=ra)
    assert [r["skipped"] for r in ores] == [r["skipped"] for r in ra] == [0, 1, 0]

    c2 = dataclasses.replace(c, **target)
    want = expected_shards(c, ostate, c2)
    b = State(torch, z, c2)
    try:
        ranks = [-1] if c2.stage <= 2 else list(range(c2.nd))
        for r in ranks:
            b.fill(-3.0)
            b.load(tmp_path, r)
            got = b.host()
            for rr in ([r] if r >= 0 else range(c2.nd)):
                mp = index_map(c2.nd, unit_lens(c2), rr)
                lo = 0 if r >= 0 else rr * mp.size
                for k in range(4):
                    g = got[k][lo:lo + mp.size]
                    # parity: the oracle's state, regrouped by the oracle
                    w = want[k][rr]
                    if k < 3:
                        assert H.rel_err(g, w) <= H.REL_STATE, (rr, k)
                    else:
                        assert H.ulp16(g, w) <= H.ULP_PARAM, (rr, k)
                    # the load moved the saved bytes exactly; padding is zero
                    valid = mp >= 0
                    assert np.array_equal(g[valid].view(np.uint8),
                                          saved[k][mp[valid]].view(np.uint8)), (rr, k)
                    assert not g[~valid].view(np.uint8).any(), (rr, k)
        r0 = z.zero_step_result(b.plan)
        assert r0["t"] == 2 and r0["loss_scale"] == scale
        if c2.stage <= 2:
            # two more steps at the new rank count, against the oracle doing the same
            rb, _ = run_steps(b, c2, (4, 5), scale)
            ores2 = oracle_steps(c2, (4, 5), ostate, osc, follow=rb)
            H.compare_runs(H.Run(*flat_of(c2, b.host()), rb), H.Run(*ostate, ores2),
                           what=f"after reshard to {target}")
    finally:
        b.close()


def test_zero3_ranks_save_and_load_as_stage2(env, tmp_path):
    """Each rank of a ZeRO-3 plan (Nd = 4, one unit per tensor) steps its own
    shard and saves its own file; a stage-2 plan at Nd = 3 loads the whole model
    and matches the oracle's flat run."""
    torch, z = env
    c3 = dataclasses.replace(BASE, nd=4, stage=3, dtype=gen.BF16, loss_scale=1.0,
                             dynamic_scale=0, inf_steps=(), steps=2, grad_sigma=1e-2)
    lens = unit_lens(c3)
    init = flat_init(c3)
    for r in range(c3.nd):
        st = State(torch, z, c3)
        try:
            mp = index_map(c3.nd, lens, r)
            valid = mp >= 0
            x = np.zeros(mp.size, np.float32)
            x[valid] = init[mp[valid]]
            st.master.copy_(torch.from_numpy(x))
            for k in (1, 2):
                G = H.grads_for_step(c3, k, c3.psi, c3.psi, 1.0)
                g = np.zeros((c3.nd, mp.size), np.uint16)
                g[:, valid] = G[:, mp[valid]]
                st.step(g)
            st.save(tmp_path, r)
        finally:
            st.close()
    ostate = [init.copy(), np.zeros(c3.psi, np.float32), np.zeros(c3.psi, np.float32),
              np.zeros(c3.psi, np.uint16)]
    oracle_steps(c3, (1, 2), ostate, oracle.new_scalars(1.0))
    c2 = dataclasses.replace(c3, nd=3, stage=2)
    b = State(torch, z, c2)
    try:
        b.fill(5.0)
        b.load(tmp_path)
        got = flat_of(c2, b.host())
        H.assert_state_close(got, ostate, "ZeRO-3 checkpoint loaded at stage 2")
        assert not b.master[c2.psi:].any()
        assert z.zero_step_result(b.plan)["t"] == 2
    finally:
        b.close()


# ------------------------------------------------------------------ failures
def small_case():
    return H.Case(shapes=[(200_001,), (4096,)], nd=4, steps=1)


def saved_small(torch, z, d, steps=(1,)):
    c = small_case()
    st = State(torch, z, c)
    try:
        st.master[:c.psi] = torch.from_numpy(flat_init(c)).cuda()
        run_steps(st, c, steps, 1.0)
        st.save(d)
    finally:
        st.close()
    return c


def untouched(st):
    return (bool((st.master == 9.0).all()) and bool((st.m == 9.0).all()) and
            bool((st.v == 9.0).all()))


def test_missing_rank_file_fails_explicitly(env, tmp_path):
    torch, z = env
    c = saved_small(torch, z, tmp_path)
    os.remove(tmp_path / "shard_00002_of_00004.zck")
    for nd in (4, 2, 8):                             # any target layout
        st = State(torch, z, dataclasses.replace(c, nd=nd))
        try:
            st.fill(9.0)
            with pytest.raises(z.ZeroError) as e:
                st.load(tmp_path)
            assert e.value.code == z.ZERO_ENOENT
            assert untouched(st)
            run_steps(st, c if nd == 4 else dataclasses.replace(c, nd=nd), (1,), 1.0)  # usable
        finally:
            st.close()


def test_missing_manifest_fails(env, tmp_path):
    torch, z = env
    c = saved_small(torch, z, tmp_path)
    os.remove(tmp_path / "manifest.zck")
    st = State(torch, z, c)
    try:
        with pytest.raises(z.ZeroError) as e:
            st.load(tmp_path)
        assert e.value.code == z.ZERO_ENOENT
        with pytest.raises(z.ZeroError) as e:
            st.load(tmp_path / "does_not_exist")
        assert e.value.code == z.ZERO_ENOENT
    finally:
        st.close()


def test_truncated_file_is_refused_before_any_write(env, tmp_path):
    torch, z = env
    c = saved_small(torch, z, tmp_path)
    p = tmp_path / "shard_00001_of_00004.zck"
    size = os.path.getsize(p)
    os.truncate(p, size - 4096)
    st = State(torch, z, c)
    try:
        st.fill(9.0)
        with pytest.raises(z.ZeroError) as e:
            st.load(tmp_path)
        assert e.value.code == z.ZERO_ECORRUPT and untouched(st)
    finally:
        st.close()


def test_damaged_block_poisons_until_a_good_load(env, tmp_path):
    torch, z = env
    c = saved_small(torch, z, tmp_path)
    p = tmp_path / "shard_00003_of_00004.zck"
    h, _, _ = read_shard(p)
    where = int(h["array_offset"][1]) + 1000          # inside m's first block
    raw = bytearray(open(p, "rb").read())
    raw[where] ^= 0x40
    open(p, "wb").write(bytes(raw))
    st = State(torch, z, c)
    try:
        with pytest.raises(z.ZeroError) as e:
            st.load(tmp_path)
        assert e.value.code == z.ZERO_ECORRUPT
        g = H.grads_for_step(c, 1, c.psi, st.padded, 1.0)
        with pytest.raises(z.ZeroError) as e:
            st.step(g)
        assert e.value.code == z.ZERO_ESTATE
        raw[where] ^= 0x40
        open(p, "wb").write(bytes(raw))
        st.load(tmp_path)
        st.step(g)
    finally:
        st.close()


def test_damaged_header_is_refused(env, tmp_path):
    torch, z = env
    c = saved_small(torch, z, tmp_path)
    p = tmp_path / "shard_00000_of_00004.zck"
    raw = bytearray(open(p, "rb").read())
    raw[4096 + 3] ^= 1                                 # the segment table
    open(p, "wb").write(bytes(raw))
    st = State(torch, z, c)
    try:
        st.fill(9.0)
        with pytest.raises(z.ZeroError) as e:
            st.load(tmp_path)
        assert e.value.code == z.ZERO_ECORRUPT and untouched(st)
    finally:
        st.close()


def test_file_from_another_step_is_refused(env, tmp_path):
    torch, z = env
    saved_small(torch, z, tmp_path / "t1", steps=(1,))
    c = saved_small(torch, z, tmp_path / "t2", steps=(1, 2))
    os.replace(tmp_path / "t1" / "shard_00001_of_00004.zck",
               tmp_path / "t2" / "shard_00001_of_00004.zck")
    st = State(torch, z, c)
    try:
        st.fill(9.0)
        with pytest.raises(z.ZeroError) as e:
            st.load(tmp_path / "t2")
        assert e.value.code == z.ZERO_ECORRUPT and untouched(st)
    finally:
        st.close()


def test_other_model_or_type_is_refused(env, tmp_path):
    torch, z = env
    c = saved_small(torch, z, tmp_path)
    for other in (dataclasses.replace(c, shapes=[(204_097,)]),           # same psi, other tensors
                  dataclasses.replace(c, dtype=gen.FP16)):
        st = State(torch, z, other)
        try:
            st.fill(9.0)
            with pytest.raises(z.ZeroError) as e:
                st.load(tmp_path)
            assert e.value.code == z.ZERO_EINVAL and untouched(st)
        finally:
            st.close()


def test_argument_checks(env, tmp_path):
    torch, z = env
    c3 = dataclasses.replace(small_case(), stage=3)
    st = State(torch, z, c3)
    try:
        for rank in (-1, 4, -2):                       # stage 3 needs one rank in range
            with pytest.raises(z.ZeroError) as e:
                st.save(tmp_path, rank)
            assert e.value.code == z.ZERO_EINVAL
        with pytest.raises(z.ZeroError):
            z.zero_checkpoint_save(st.plan, str(tmp_path), 0, st.master.data_ptr() + 4, st.m,
                                   st.v, st.params)     # misaligned
        st.save(tmp_path, 0)
        assert sorted(os.listdir(tmp_path)) == ["manifest.zck", "shard_00000_of_00004.zck"]
        with pytest.raises(z.ZeroError) as e:           # ranks 1-3 never saved
            st.load(tmp_path, 0)
        assert e.value.code == z.ZERO_ENOENT
    finally:
        st.close()


# ---------------------------------------------------------- full size (GPT-2 small)
def test_gpt2_small_full_size_reshard_round_trip(env, tmp_path):
    """All 124 M parameters, Nd = 8 -> 4 and back to 8 through two
    checkpoints (fsync'd): every byte comes back, padding zeroed."""
    from gen import workloads as W
    torch, z = env
    w = W.gpt2_small()
    c = H.from_workload(w)
    a = State(torch, z, c)
    try:
        gen.cuda_f32(a.master.data_ptr(), c.seed, gen.STREAM_MASTER, 0, 0, c.psi, 0.02)
        a.m.normal_()
        a.v.uniform_()
        a.params.random_(-32768, 32767)
        a.master[c.psi:] = 0
        a.m[c.psi:] = 0
        a.v[c.psi:] = 0
        a.params[c.psi:] = 0
        a.save(tmp_path / "nd8", flags=z.ZERO_CKPT_FSYNC)
        before = a.host()
    finally:
        a.close()
    b = State(torch, z, dataclasses.replace(c, nd=4))
    try:
        b.fill(1.0)
        b.load(tmp_path / "nd8")
        mid = b.host()
        for x, y in zip(before, mid):
            assert np.array_equal(x[:c.psi].view(np.uint8), y[:c.psi].view(np.uint8))
            assert not y[c.psi:].view(np.uint8).any()
        b.save(tmp_path / "nd4")
    finally:
        b.close()
    a = State(torch, z, c)
    try:
        a.fill(2.0)
        a.load(tmp_path / "nd4")
        for x, y in zip(before, a.host()):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
    finally:
        a.close()
