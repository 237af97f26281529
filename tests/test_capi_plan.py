"""The C-ABI library loads, exports every declared symbol, and its planner
matches the oracle planner table for table, bit for bit (CPU only)."""
import os
import re

import numpy as np
import pytest

import synth
from oracle import plan as oplan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import prefix_tree_packed_gb300 as lib
    return lib


def test_exports_every_declared_symbol(lib):
    declared = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            with open(os.path.join(ROOT, "include", h)) as f:
                declared |= set(re.findall(r"^TREE_API\s+[\w\s\*]*?\*?\s*(\w+)\s*\(", f.read(), flags=re.M))
    assert declared == set(lib.EXPORTS)
    for name in declared:
        getattr(lib._lib, name)          # raises if the shared object lacks it
    assert lib.version() >= 100


def _compare(p_or: oplan.Plan, q_or: dict, pl):
    t = pl.tables()
    i = pl.info
    assert (i.n_blocks, i.n_tot, i.n_res, i.n_chunks, i.n_slots) == (
        p_or.n_blocks, p_or.n_tot, p_or.n_res, p_or.n_chunks, p_or.n_slots)
    assert i.pairs == p_or.pairs
    pairs = [("block_map", p_or.block_map), ("blk_start", p_or.blk_start), ("blk_len", p_or.blk_len),
             ("blk_parent", p_or.blk_parent), ("blk_depth", p_or.blk_depth), ("blk_pos0", p_or.blk_pos0),
             ("blk_send", p_or.blk_send), ("blk_resident", p_or.blk_resident), ("blk_slot", p_or.blk_slot),
             ("pos", p_or.pos), ("send", p_or.send), ("chunk_q0", p_or.chunk_q0), ("chunk_q1", p_or.chunk_q1),
             ("chunk_t0", p_or.chunk_t0), ("chunk_t1", p_or.chunk_t1), ("qt_row0", p_or.qt_row0),
             ("qt_row1", p_or.qt_row1), ("qt_ent0", p_or.qt_ent0), ("qt_ent1", p_or.qt_ent1),
             ("ent", p_or.ent), ("qt_order", p_or.qt_order), ("slot_tok", p_or.slot_tok)]
    if q_or:
        pairs += [("r1", q_or["r1"]), ("r2", q_or["r2"])]
    for name, ref in pairs:
        assert np.array_equal(t[name].astype(np.int64), np.asarray(ref, np.int64)), name
    assert i.max_pos == int(p_or.pos.max()) + 1
    for c in range(i.n_chunks):
        ci = pl.chunk(c)
        q0, q1 = int(p_or.chunk_q0[c]), int(p_or.chunk_q1[c])
        assert ci.pairs == int((p_or.pos[q0:q1] + 1).sum())
    # the device image holds the same arrays at the advertised offsets
    img = t["image"].view(np.int32)
    assert np.array_equal(img[i.off_pos // 4: i.off_pos // 4 + i.n_tot], t["pos"])
    assert np.array_equal(img[i.off_send // 4: i.off_send // 4 + len(t["send"])], t["send"])
    qt = img[i.off_qtile // 4: i.off_qtile // 4 + 4 * i.n_qtiles].reshape(-1, 4)
    assert np.array_equal(qt[:, 0], t["qt_row0"]) and np.array_equal(qt[:, 3], t["qt_ent1"])
    assert np.array_equal(img[i.off_ent // 4: i.off_ent // 4 + i.n_entries], t["ent"])
    assert np.array_equal(img[i.off_order // 4: i.off_order // 4 + i.n_qtiles], t["qt_order"])
    for off in (i.off_pos, i.off_send, i.off_qtile, i.off_ent, i.off_order, i.off_chunk, i.off_slot_tok,
                i.off_r1, i.off_r2):
        assert off % 16 == 0


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_workloads_match_oracle(lib, n):
    w = synth.workload(n)
    f = w.forest
    kw = dict(leaf1=w.leaf1, leaf2=w.leaf2) if w.leaf1 is not None else {}
    p_or, q_or = oplan.plan_forest(f, max_fwd=w.max_fwd, **kw)
    pl = lib.Plan.from_forest(f, max_fwd=w.max_fwd, **kw)
    _compare(p_or, q_or, pl)


@pytest.mark.parametrize("seed", range(40))
def test_random_forests_match_oracle(lib, seed):
    rng = np.random.default_rng(1000 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 5)), max_blocks=int(rng.integers(2, 40)),
                            max_len=int(rng.integers(1, 300)), dup_prob=0.25, resident_root=bool(seed % 4 == 0))
    max_fwd = int(rng.choice([128, 256, 8192]))
    try:
        p_or, _ = oplan.plan_forest(f, max_fwd=max_fwd)
    except oplan.PlanError as e:
        with pytest.raises(lib.TreeError) as ei:
            lib.Plan.from_forest(f, max_fwd=max_fwd)
        assert ei.value.code == e.code
        return
    pl = lib.Plan.from_forest(f, max_fwd=max_fwd)
    _compare(p_or, {}, pl)


def test_error_codes_match_oracle(lib):
    cases = [
        ([-1] + list(range(8)), [1] * 9, None, {}),           # depth 9
        ([-1], [32769], None, {}),                             # row too long
        ([-1, 0, 0], [20000, 10000, 3000], None, {}),          # row too long across blocks
        ([-1, 2, 1], [1, 1, 1], None, {}),                     # cycle
        ([-1, 5], [1, 1], None, {}),                           # orphan
        ([-1, 0], [1, 0], None, {}),                           # empty block
        ([-1, 0], [1, -3], None, {}),                          # negative length
        ([-1, -1], [4, 4], [0, 1], {}),                        # resident after a forward block
        ([-1], [4], [1], {}),                                  # nothing to compute
        ([-1], [4], None, {"max_fwd": 100}),                   # chunk not a multiple of 128
    ]
    for par, ln, res, kw in cases:
        with pytest.raises(oplan.PlanError) as eo:
            oplan.make_plan(par, ln, np.zeros(len(par), np.uint64), res or [0] * len(par), **kw)
        with pytest.raises(lib.TreeError) as ec:
            lib.Plan(par, ln, None, res, **kw)
        assert ec.value.code == eo.value.code, (par, ln, res, kw)
        assert str(ec.value)


def test_question_errors(lib):
    # a question naming a non-leaf block
    with pytest.raises(lib.TreeError) as e:
        lib.Plan([-1, 0, 0], [4, 2, 2], leaf1=[0], leaf2=[1])
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError):
        lib.Plan([-1, 0, 0], [4, 2, 2], leaf1=[1], leaf2=[7])


def _check_runs(runs, send, rng):
    """Run tables against maximal runs of equal send recomputed from the oracle's send."""
    n_kvt = runs.shape[0]
    for t in range(n_kvt):
        sd = send[128 * t: 128 * t + 128]
        starts = [0] + [c for c in range(1, 128) if sd[c] != sd[c - 1]]
        n = int(runs[t, 0])
        assert n == len(starts)
        if n > 16:
            assert not runs[t, 1:].any()
            continue
        assert not runs[t, 1:4].any()
        masks = []
        for r, a in enumerate(starts):
            b = starts[r + 1] if r + 1 < n else 128
            assert runs[t, 4 + r] == sd[a]
            bits = runs[t, 20 + 4 * r: 24 + 4 * r].astype(np.uint32)
            m = np.array([(int(bits[c // 32]) >> (c % 32)) & 1 for c in range(128)], bool)
            assert np.array_equal(m, (np.arange(128) >= a) & (np.arange(128) < b))
            masks.append(m)
        assert not runs[t, 4 + n: 20].any() and not runs[t, 20 + 4 * n:].any()
        # what the kernel relies on: OR of the runs that end after a query = the key-by-key test
        for i in rng.integers(0, int(sd.max()) + 2, 8):
            vis = np.zeros(128, bool)
            for r in range(n):
                if i < runs[t, 4 + r]:
                    vis |= masks[r]
            assert np.array_equal(vis, i < sd)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5])
def test_run_tables_workloads(lib, n):
    w = synth.workload(n)
    kw = dict(leaf1=w.leaf1, leaf2=w.leaf2) if w.leaf1 is not None else {}
    plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd, **kw)
    ref, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd, **kw)
    send = np.zeros(plan.tables()["runs"].shape[0] * 128, np.int64)
    rs = np.asarray(ref.send)[: len(send)]  # the oracle's send (0 past n_tot)
    send[: len(rs)] = rs
    _check_runs(plan.tables()["runs"], send, np.random.default_rng(n))


@pytest.mark.parametrize("seed", range(6))
def test_run_tables_random_forests(lib, seed):
    rng = np.random.default_rng(700 + seed)
    # tiny blocks give tiles of more than 16 runs, larger ones fewer
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(10, 90)),
                            max_len=[3, 6, 40][seed % 3], resident_root=bool(seed % 2))
    try:
        ref, _ = oplan.plan_forest(f, max_fwd=8192)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    plan = lib.Plan.from_forest(f, max_fwd=8192)
    runs = plan.tables()["runs"]
    send = np.zeros(runs.shape[0] * 128, np.int64)
    rs = np.asarray(ref.send)[: len(send)]
    send[: len(rs)] = rs
    _check_runs(runs, send, rng)


def test_upload_argument_checks(lib):
    # every check runs before any CUDA call, so no device is needed
    plan = lib.Plan([-1, 0, 0], [130, 7, 9])
    need = plan.info.dev_bytes
    with pytest.raises(lib.TreeError) as e:
        plan.upload_staged(16, need, 32, need - 4)          # staging too small
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        plan.upload_staged(16, need - 4, 32, need)          # device buffer too small
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        plan.upload_staged(16, need, 0, need)               # no staging buffer
    assert e.value.code == lib.TREE_ERR_INVALID_ARG
    with pytest.raises(lib.TreeError) as e:
        plan.upload_staged(24, need, 32, need)              # misaligned device buffer
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED
    with pytest.raises(lib.TreeError) as e:
        plan.upload(24, need)
    assert e.value.code == lib.TREE_ERR_UNSUPPORTED


def test_rope_table_matches_double_precision(lib):
    tab = lib.rope_table(40000, 128, 500000.0)
    from oracle import rope
    a = rope.angles(np.arange(40000), 128, 500000.0)
    # both evaluate in double and round once to float: at most one float ulp apart
    # (the two libraries' pow/cos/sin may differ in the last double bit)
    np.testing.assert_array_max_ulp(tab[..., 0], np.cos(a).astype(np.float32), maxulp=1)
    np.testing.assert_array_max_ulp(tab[..., 1], np.sin(a).astype(np.float32), maxulp=1)
    with pytest.raises(lib.TreeError):
        lib.rope_table(0, 64, 1e4)


# ---------------------------------------------------------------- tiling by position

def _position_tiles_of(plan, t_):
    """Per forward row: list of (entry order, position tile, {slot: key}) the row takes its keys from."""
    i = plan.info
    out = {}
    vk, vr = t_["vkeys"], t_["vruns"]
    for q in range(i.n_qtiles):
        r0, r1 = int(t_["qt_row0"][q]), int(t_["qt_row1"][q])
        for k, e in enumerate(range(int(t_["qt_ent0"][q]), int(t_["qt_ent1"][q]))):
            ev = int(t_["ent"][e])
            if ev & 3 == 2:   # full and contiguous: names its first key
                assert ev >> 2 == vk[e][0]
            else:
                assert ev >> 2 == e
            run = vr[e]
            n = int(run[0])
            rows = run[4:8].astype(np.uint32)
            if ev & 2:   # contiguous: one tiled box of consecutive keys
                assert (vk[e] == vk[e][0] + np.arange(128)).all()
            full = not (ev & 1)
            for row in range(r1 - r0):
                if not (rows[row >> 5] >> (row & 31)) & 1:
                    continue
                iq = r0 + row
                seen = {}
                for rr in range(n):
                    c0, c1, j0, se = (int(x) for x in run[8 + 4 * rr: 12 + 4 * rr])
                    assert (vk[e][c0:c1 + 1] == np.arange(j0, j0 + c1 - c0 + 1)).all()
                    if not (j0 <= iq < se):
                        continue
                    for c in range(c0, min(c1, c0 + iq - j0) + 1):
                        assert c not in seen
                        seen[c] = j0 + c - c0
                if full:   # no mask: every row of the tile is served and sees every slot
                    assert len(seen) == 128
                out.setdefault(iq, []).append((k, seen))
            if full:
                assert all((rows[x >> 5] >> (x & 31)) & 1 for x in range(r1 - r0))
    return out


def _check_position_tiling(plan, mask):
    t_ = plan.tables()
    i = plan.info
    pos = t_["pos"]
    per_row = _position_tiles_of(plan, t_)
    for iq in range(i.n_res, i.n_tot):
        got = {}
        tiles = []
        for k, seen in per_row.get(iq, []):
            if not seen:
                continue
            ts = {int(pos[j]) // 128 for j in seen.values()}
            assert len(ts) == 1               # one position range per entry
            t = ts.pop()
            tiles.append(t)
            for c, j in seen.items():
                assert c == int(pos[j]) % 128  # key at position p in slot p % 128
                assert j not in got            # each key once
                got[j] = c
        assert tiles == sorted(tiles) and len(set(tiles)) == len(tiles)
        want = set(np.nonzero(mask[iq])[0].tolist())
        assert set(got) == want, iq


@pytest.mark.parametrize("seed", range(8))
def test_position_tiling_random_forests(lib, seed):
    rng = np.random.default_rng(900 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(4, 40)),
                            max_len=[3, 9, 60, 200][seed % 4], resident_root=bool(seed % 2))
    try:
        ref, _ = oplan.plan_forest(f, max_fwd=8192)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    plan = lib.Plan.from_forest(f, max_fwd=8192, tiling=1)
    assert plan.info.tiling == 1
    # same packing as the packed tiling
    t0 = lib.Plan.from_forest(f, max_fwd=8192).tables()
    np.testing.assert_array_equal(plan.tables()["pos"], t0["pos"])
    _check_position_tiling(plan, oplan.brute_mask(ref))


def test_position_tiling_workload1_and_alone_equals_packed(lib):
    w = synth.workload(1)
    ref, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd)
    plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd, tiling=1)
    _check_position_tiling(plan, oplan.brute_mask(ref))
    # one prompt alone: the position tiles are the packed tiles (packed index = position)
    alone = lib.Plan([-1, 0], [200, 90], tiling=1)
    t_ = alone.tables()
    assert alone.info.n_entries == lib.Plan([-1, 0], [200, 90]).info.n_entries
    for e in range(alone.info.n_entries):
        run = t_["vruns"][e]
        assert run[0] >= 1
    assert lib.Plan([-1], [10], tiling=1).info.n_entries == 1
    with pytest.raises(lib.TreeError):
        lib.Plan([-1], [10], tiling=3)


# ---------------------------------------------------------------- gathered key tiles

def _check_gathered_tiling(plan, mask, bm):
    """Every row of a query tile takes exactly its visible keys from the tile's gathered
    entries, each once; an entry holds keys nobody in the tile sees only in slots no run covers."""
    t_ = plan.tables()
    i = plan.info
    assert i.tiling == 2 and i.bm == bm
    send = t_["send"]
    r0s, r1s = t_["qt_row0"], t_["qt_row1"]
    # query tiles of bm tokens cover every forward row once, chunk by chunk
    rows = np.concatenate([np.arange(a, b) for a, b in zip(r0s, r1s)])
    np.testing.assert_array_equal(np.sort(rows), np.arange(i.n_res, i.n_tot))
    assert all(b - a <= bm for a, b in zip(r0s, r1s))
    per_row = _position_tiles_of(plan, t_)
    vk, vr = t_["vkeys"], t_["vruns"]
    for q in range(i.n_qtiles):
        r0, r1 = int(r0s[q]), int(r1s[q])
        prev = -1
        union = set()
        for e in range(int(t_["qt_ent0"][q]), int(t_["qt_ent1"][q])):
            run = vr[e]
            n = int(run[0])
            assert 1 <= n <= 16
            # every row of the tile is assigned to every entry
            assert all((int(run[4 + (x >> 5)]) >> (x & 31)) & 1 for x in range(r1 - r0))
            for rr in range(n):
                c0, c1, j0, se = (int(x) for x in run[8 + 4 * rr: 12 + 4 * rr])
                assert c0 <= c1 and j0 > prev          # keys ascend through the tile's entries
                if rr == 0 or j0 != prev + 1:          # a stretch of consecutive keys starts on 8 slots
                    assert c0 % 8 == 0
                else:                                  # else it continues the run before, slot by slot
                    assert c0 == int(run[8 + 4 * (rr - 1) + 1]) + 1
                prev = j0 + c1 - c0
                assert (send[j0:prev + 1] == se).all()  # one subtree end: one block's piece
                union.update(range(j0, prev + 1))
        want = set()
        for iq in range(r0, r1):
            want |= set(np.nonzero(mask[iq])[0].tolist())
        assert union == want, q                         # no key that nobody in the tile sees
    for iq in range(i.n_res, i.n_tot):
        got = []
        for _, seen in per_row.get(iq, []):
            got += list(seen.values())
        assert len(got) == len(set(got))                # each key once
        assert set(got) == set(np.nonzero(mask[iq])[0].tolist()), iq


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("pack", [1, 4])
def test_gathered_tiling_random_forests(lib, seed, pack):
    rng = np.random.default_rng(1300 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(4, 40)),
                            max_len=[3, 9, 60, 200][seed % 4], resident_root=bool(seed % 2))
    try:
        ref, _ = oplan.plan_forest(f, max_fwd=1024)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    plan = lib.Plan.from_forest(f, max_fwd=1024, tiling=2, pack_heads=pack)
    assert plan.info.pack_heads == pack
    t0 = lib.Plan.from_forest(f, max_fwd=1024).tables()
    np.testing.assert_array_equal(plan.tables()["pos"], t0["pos"])  # same packing
    _check_gathered_tiling(plan, oplan.brute_mask(ref), 256 // pack if pack > 1 else 128)


@pytest.mark.parametrize("pack", [2, 8])
def test_gathered_tiling_many_tiny_blocks(lib, pack):
    # a bush of one-token leaves: more than 16 blocks reach into one query tile, so entries split at 16 runs
    parent = [-1] + [0] * 300
    length = [40] + [1] * 300
    f = synth.Forest(np.array(parent, np.int32), np.array(length, np.int32), np.arange(1, 302, dtype=np.uint64),
                     np.zeros(301, np.uint8))
    ref, _ = oplan.plan_forest(f, max_fwd=8192)
    plan = lib.Plan.from_forest(f, tiling=2, pack_heads=pack)
    _check_gathered_tiling(plan, oplan.brute_mask(ref), 256 // pack)


def test_gathered_tiling_small_leaves_one_entry_per_tile(lib):
    # many short prompts under a shared template: with four heads packed, each 64-token query tile
    # sees the template and at most 64 + 23 keys of its own leaves: one gathered tile
    w = synth.workload(5)
    plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd, tiling=2, pack_heads=4)
    i = plan.info
    assert i.bm == 64 and i.n_entries == i.n_qtiles
    packed = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd).info
    # the same visible pairs for a third of the MMA tiles: per kv head, a packed entry is met by
    # each of the 4 q heads, a gathered one by the tile's two halves (4 heads x 32 tokens each)
    assert i.pairs == packed.pairs
    assert i.n_entries * 2 * 2.5 < packed.n_entries * 4


def test_gathered_tiling_options_checked(lib):
    with pytest.raises(lib.TreeError):
        lib.Plan([-1], [10], tiling=2, pack_heads=3)
    with pytest.raises(lib.TreeError):
        lib.Plan([-1], [10], tiling=0, pack_heads=4)
    assert lib.Plan([-1], [10], tiling=1, pack_heads=2).info.bm == 128
    assert lib.Plan([-1], [10], tiling=2, pack_heads=1).info.bm == 128


@pytest.mark.parametrize("seed", range(4))
def test_position_tiling_packed_heads_random_forests(lib, seed):
    # query tiles of 256 / R tokens; every row still takes its keys per position range from one entry
    rng = np.random.default_rng(1900 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(4, 40)),
                            max_len=[3, 9, 60, 200][seed % 4], resident_root=bool(seed % 2))
    try:
        ref, _ = oplan.plan_forest(f, max_fwd=8192)
    except oplan.PlanError:
        pytest.skip("forest has no forward tokens")
    R = [2, 4, 8, 4][seed]
    plan = lib.Plan.from_forest(f, max_fwd=8192, tiling=1, pack_heads=R)
    assert plan.info.bm == 256 // R and plan.info.pack_heads == R
    _check_position_tiling(plan, oplan.brute_mask(ref))
