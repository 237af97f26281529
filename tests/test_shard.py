"""Rows of one batch shared out over ranks (tree_shard_rows / tree_shard_select), on CPU.

Rows are independent trees (a query sees only its own prompt), so a batch can be split by rows
over GPUs with the resident template kept everywhere and the decisions gathered on the host.
Checked here:
  * the library's split equals the rule restated below in plain Python from the oracle's plan
    (rows after merging, units joined by questions, cost = visible pairs, longest first to the
    least-loaded rank), on every workload and on random forests;
  * each rank's share plans to the same prompts: every question's readout token has the same
    position and content on its rank as in the whole batch;
  * two gloo ranks, each running the oracle on its share and gathering its decisions, reproduce
    the decisions of the whole batch computed in one place, exactly.
"""
import os
import socket
import sys

import numpy as np
import pytest

import synth
from oracle import attention as oatt
from oracle import plan as oplan
from oracle import readout as ordo
from oracle import rope as orope

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import prefix_tree_packed_gb300 as lib
    return lib


def lpt_by_hand(p, leaf1, leaf2, n_ranks):
    """The split rule from its statement, over the oracle plan's merged blocks."""
    row = {}
    for b in range(p.n_blocks):                       # packed order: parents first
        if p.blk_resident[b]:
            continue
        par = int(p.blk_parent[b])
        row[b] = b if par < 0 or p.blk_resident[par] else row[par]
    cost = {}
    for b, r in row.items():
        L, p0 = int(p.blk_len[b]), int(p.blk_pos0[b])
        cost[r] = cost.get(r, 0) + L * p0 + L * (L + 1) // 2
    unit = {r: r for r in cost}                       # union of rows joined by a question

    def find(x):
        while unit[x] != x:
            x = unit[x]
        return x
    for a, c in zip(leaf1, leaf2):
        ra, rc = find(row[int(p.block_map[a])]), find(row[int(p.block_map[c])])
        if ra != rc:
            unit[max(ra, rc)] = min(ra, rc)
    ucost = {}
    for r in sorted(cost):
        ucost[find(r)] = ucost.get(find(r), 0) + cost[r]
    order = sorted(ucost, key=lambda u: (-ucost[u], u))
    load = [0] * n_ranks
    urank = {}
    for u in order:
        k = min(range(n_ranks), key=lambda i: (load[i], i))
        urank[u] = k
        load[k] += ucost[u]
    block_rank = np.array([-1 if p.blk_resident[int(p.block_map[i])] else urank[find(row[int(p.block_map[i])])]
                           for i in range(len(p.block_map))], np.int32)
    q_rank = np.array([urank[find(row[int(p.block_map[a])])] for a in leaf1], np.int32)
    return block_rank, q_rank, np.array(load, np.int64), max(ucost.values(), default=0)


def _questions(f, rng, n_q):
    """Questions over random pairs of leaves of the same tree or of sibling trees."""
    nb = len(f.parent)
    has_child = np.zeros(nb, bool)
    has_child[f.parent[f.parent >= 0]] = True
    leaves = np.nonzero(~has_child & (f.resident == 0))[0]
    if len(leaves) == 0:
        return None, None
    return rng.choice(leaves, n_q).astype(np.int32), rng.choice(leaves, n_q).astype(np.int32)


def _cases():
    for n in (1, 2, 3, 4, 5):
        w = synth.workload(n)
        yield f"workload{n}", w.forest, w.leaf1, w.leaf2, w.max_fwd
    for s in range(12):
        rng = np.random.default_rng(70 + s)
        f = synth.random_forest(rng, n_roots=int(rng.integers(1, 5)), max_blocks=int(rng.integers(4, 40)),
                                max_len=int(rng.integers(1, 120)), dup_prob=0.25, resident_root=bool(s % 2))
        l1, l2 = _questions(f, rng, int(rng.integers(1, 6)))
        yield f"random{s}", f, l1, l2, 8192


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 5])
def test_split_equals_the_rule(lib, n_ranks):
    for name, f, l1, l2, max_fwd in _cases():
        kw = dict(leaf1=l1, leaf2=l2) if l1 is not None else {}
        try:
            p, _ = oplan.plan_forest(f, max_fwd=max_fwd, **kw)
        except oplan.PlanError:
            continue
        spec = lib.Spec.from_forest(f, max_fwd=max_fwd, **kw)
        br, qr, pairs = lib.shard_rows(spec, n_ranks)
        wb, wq, wp, biggest = lpt_by_hand(p, l1 if l1 is not None else [], l2 if l2 is not None else [], n_ranks)
        assert np.array_equal(br, wb), name
        assert np.array_equal(qr, wq), name
        assert np.array_equal(pairs, wp), name
        assert pairs.sum() == p.pairs, name            # every visible pair lands on exactly one rank
        if l1 is not None:                             # a question's two leaves share its rank
            assert np.array_equal(br[l1], qr) and np.array_equal(br[l2], qr), name
        # longest first: no rank exceeds the least loaded one by more than the largest unit
        assert pairs.max() - pairs.min() <= biggest, name


def test_split_balances_the_llama1b_rows(lib):
    w = synth.workload(2)
    spec = lib.Spec.from_forest(w.forest, leaf1=w.leaf1, leaf2=w.leaf2)
    for n in (1, 2, 4, 8):
        br, qr, pairs = lib.shard_rows(spec, n)
        assert len(set(pairs.tolist())) == 1             # 8 identical rows: equal shares
        assert np.bincount(qr, minlength=n).tolist() == [32 // n] * n


def test_question_joining_rows_keeps_them_together(lib):
    # two roots, one question reading a leaf of each: one unit, one rank
    parent, length = [-1, 0, -1, 2, -1], [10, 5, 12, 5, 40]
    spec = lib.Spec(parent, length, leaf1=[1], leaf2=[3])
    br, qr, pairs = lib.shard_rows(spec, 2)
    assert br[0] == br[1] == br[2] == br[3] == qr[0]
    assert br[4] != br[0]


def test_split_rejects_bad_arguments(lib):
    spec = lib.Spec([-1, 0], [8, 4], resident=[1, 0], leaf1=[0], leaf2=[1])
    with pytest.raises(lib.TreeError):
        lib.shard_rows(spec, 2)                          # a question reads out the resident block
    spec = lib.Spec([-1, 0], [8, 4])
    with pytest.raises(lib.TreeError):
        lib.shard_rows(spec, 0)


def _token_content(p, gblock_of_packed, seed, hq, hkv, d):
    """Q/K/V of every packed token, drawn per merged block of the whole batch (so a token has the
    same values however the batch is split)."""
    q = np.empty((p.n_tot, hq, d), np.float16)
    k = np.empty((p.n_tot, hkv, d), np.float16)
    v = np.empty((p.n_tot, hkv, d), np.float16)
    for b in range(p.n_blocks):
        s, L = int(p.blk_start[b]), int(p.blk_len[b])
        r = np.random.default_rng(seed * 100003 + int(gblock_of_packed[b]))
        q[s:s + L] = r.standard_normal((L, hq, d)).astype(np.float16)
        k[s:s + L] = r.standard_normal((L, hkv, d)).astype(np.float16)
        v[s:s + L] = r.standard_normal((L, hkv, d)).astype(np.float16)
    return q, k, v


def _decide(forest, leaf1, leaf2, n_letters, temps, gblock_of_input, seed, hq=4, hkv=2, d=64, stride=6):
    """Oracle decisions of a batch: attention of the readout tokens, letter logits taken from their
    outputs, readout and calibration.  Returns p_cal [n_q, stride], choice [n_q], slot positions."""
    p, qm = oplan.plan_forest(forest, leaf1=leaf1, leaf2=leaf2)
    gpk = np.empty(p.n_blocks, np.int64)
    gpk[p.block_map] = np.asarray(gblock_of_input)      # merged blocks hold identical input blocks
    q, k, v = _token_content(p, gpk, seed, hq, hkv, d)
    qr, kr = orope.apply_plan(p, q[p.n_res:], k, 500000.0)
    rows = np.asarray(p.slot_tok) - p.n_res
    o = oatt.attend_rows(p, qr, kr, v, rows)
    logits = (3.0 * o[:, 0, :stride]).astype(np.float32)
    pc, _, _ = ordo.decide(logits, qm["r1"], qm["r2"], n_letters, temps, stride)
    ch = ordo.choice_f32(logits, qm["r1"], qm["r2"], n_letters)
    pos = p.pos[np.asarray(p.slot_tok)][qm["r1"]], p.pos[np.asarray(p.slot_tok)][qm["r2"]]
    return pc, ch, np.stack(pos, 1)


def _batch():
    rng = np.random.default_rng(5)
    b = synth._Builder()
    t = b.add(-1, 24, key=1, resident=1)
    l1, l2 = [], []
    for r in range(6):
        doc = b.add(t, int(rng.integers(20, 60)))
        for _ in range(int(rng.integers(1, 3))):
            qb = b.add(doc, int(rng.integers(5, 15)))
            l1.append(b.add(qb, int(rng.integers(3, 9))))
            l2.append(b.add(qb, int(rng.integers(3, 9))))
    # a question whose two leaves are separate rows under the template
    l1.append(b.add(t, 7))
    l2.append(b.add(t, 9))
    f = b.forest()
    nq = len(l1)
    return f, np.array(l1, np.int32), np.array(l2, np.int32), rng.integers(2, 7, nq).astype(np.int32), \
        rng.choice([0.5, 1.0, 2.0], nq).astype(np.float32)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import prefix_tree_packed_gb300 as lib
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        f, l1, l2, nl, T = _batch()
        spec = lib.Spec.from_forest(f, leaf1=l1, leaf2=l2)
        br, qr, _ = lib.shard_rows(spec, world)
        sel = lib.shard_select(spec, br, qr, rank)
        sub = synth.Forest(sel["parent"], sel["length"], sel["key"], sel["resident"])
        qi = sel["question_index"]
        gp, _ = oplan.plan_forest(f, leaf1=l1, leaf2=l2)
        gblock = gp.block_map[sel["block_index"]]        # merged block of the whole batch
        pc, ch, pos = _decide(sub, sel["leaf1"], sel["leaf2"], nl[qi], T[qi], gblock, seed=9)
        # the library plans the share like the oracle: same readout slots
        plan = lib.Plan.from_forest(sub, leaf1=sel["leaf1"], leaf2=sel["leaf2"])
        tb = plan.tables()
        _, qm = oplan.plan_forest(sub, leaf1=sel["leaf1"], leaf2=sel["leaf2"])
        same_slots = np.array_equal(tb["r1"], qm["r1"]) and np.array_equal(tb["r2"], qm["r2"])
        gathered = [None] * world
        dist.all_gather_object(gathered, (qi, pc, ch, pos, same_slots))
        out.put((rank, gathered))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gather_the_decisions_of_the_whole_batch():
    import torch.multiprocessing as mp
    f, l1, l2, nl, T = _batch()
    gp, _ = oplan.plan_forest(f, leaf1=l1, leaf2=l2)
    want_pc, want_ch, want_pos = _decide(f, l1, l2, nl, T, gp.block_map, seed=9)
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=300) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, gathered in res:
        got_pc = np.full_like(want_pc, np.nan)
        got_ch = np.full_like(want_ch, -5)
        got_pos = np.full_like(want_pos, -5)
        seen = np.zeros(len(l1), int)
        for qi, pc, ch, pos, same_slots in gathered:
            assert same_slots
            assert len(qi) > 0                           # both ranks answer questions
            got_pc[qi], got_ch[qi], got_pos[qi] = pc, ch, pos
            seen[qi] += 1
        assert (seen == 1).all()                         # every question answered by exactly one rank
        assert np.array_equal(got_pos, want_pos)         # readout tokens at the same prompt positions
        assert np.array_equal(got_ch, want_ch)
        assert np.array_equal(got_pc, want_pc)           # bit for bit: each row's prompt is the same
