"""Pins for the oracle planner (CPU only).

Checks the packing against the page's token-count example, against brute
force visibility on small random forests, and the limits the page states.
"""
import json
import os

import numpy as np
import pytest

import synth
from oracle import plan as oplan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "token_counts.json")


def _six_prompt_forest(g, template_resident=True):
    parent, length, key, res = [], [], [], []

    def add(p, L, r=0):
        parent.append(p); length.append(L); key.append(0); res.append(r)
        return len(parent) - 1

    t = add(-1, g["template"], 1 if template_resident else 0)
    s = add(t, g["state"])
    leaves = []
    for _ in range(g["questions"]):
        q = add(s, g["question"])
        for _ in range(g["orders"]):
            leaves.append(add(q, g["option"]))
    return (np.array(parent), np.array(length), np.array(key, np.uint64), np.array(res)), leaves


def test_page_token_count_example():
    with open(GOLDEN) as f:
        g = json.load(f)
    (par, ln, key, res), leaves = _six_prompt_forest(g)
    p, _ = oplan.make_plan(par, ln, key, res)
    # every prompt ends at position 214: 215 tokens each
    for lf in leaves:
        b = p.block_map[lf]
        assert p.pos[p.slot_tok[p.blk_slot[b]]] + 1 == g["prompt_tokens_printed"]
    assert len(leaves) == g["prompts_printed"]
    alone = g["prompts_printed"] * g["prompt_tokens_printed"]
    assert p.n_fwd == 300
    assert round(alone / p.n_fwd, 1) == g["reduction_printed"]
    # counting the template as well gives a smaller factor than printed
    assert round(alone / p.n_tot, 1) != g["reduction_printed"]


def _check_tables_vs_brute(p):
    bm = oplan.brute_mask(p)
    assert np.array_equal(bm, oplan.mask_from_tables(p))
    # rebuild the forward rows' visibility from the tile lists alone
    rebuilt = np.zeros((p.n_fwd, p.n_tot), bool)
    for t in range(len(p.qt_row0)):
        i0, i1 = int(p.qt_row0[t]), int(p.qt_row1[t])
        for e in p.ent[p.qt_ent0[t]:p.qt_ent1[t]]:
            kt, partial = int(e) >> 1, int(e) & 1
            j0, j1 = kt * p.bn, min(kt * p.bn + p.bn, p.n_tot)
            for i in range(i0, i1):
                for j in range(j0, j1):
                    vis = True if not partial else (j <= i < p.send[j])
                    rebuilt[i - p.n_res, j] = vis
            if not partial:
                assert bm[i0:i1, j0:j1].all()
    assert np.array_equal(rebuilt, bm[p.n_res:])
    assert oplan.OK == 0
    # pairs closed form against the brute count
    assert p.pairs == int(bm[p.n_res:].sum())


@pytest.mark.parametrize("seed", range(12))
def test_random_forests_against_brute_force(seed):
    rng = np.random.default_rng(seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 4)), max_blocks=int(rng.integers(3, 16)),
                            max_len=int(rng.integers(1, 40)), resident_root=bool(seed % 3 == 0))
    try:
        p, _ = oplan.plan_forest(f, max_fwd=128)
    except oplan.PlanError as e:
        assert e.code == oplan.ERR_INVALID_ARG   # all-resident forest
        return
    _check_tables_vs_brute(p)


def test_large_random_tiles_against_brute_force():
    rng = np.random.default_rng(123)
    f = synth.random_forest(rng, n_roots=2, max_blocks=24, max_len=90, dup_prob=0.1)
    p, _ = oplan.plan_forest(f, max_fwd=256)
    assert p.n_tot > 400 and p.n_chunks >= 2
    _check_tables_vs_brute(p)


def test_workload_token_counts_and_pairs():
    p1, q1 = oplan.plan_forest(synth.workload(1).forest, leaf1=[1], leaf2=[2])
    assert (p1.n_tot, p1.n_res, p1.n_slots) == (96, 0, 2)
    assert list(q1["r1"]) == [0] and list(q1["r2"]) == [1]
    w2 = synth.workload(2)
    p2, q2 = oplan.plan_forest(w2.forest, leaf1=w2.leaf1, leaf2=w2.leaf2)
    assert (p2.n_res, p2.n_fwd, p2.n_chunks, p2.n_slots) == (128, 8192, 1, 64)
    # closed form per block: sum over its tokens of (pos + 1)
    def closed(p):
        tot = 0
        for b in range(p.n_blocks):
            if p.blk_resident[b]:
                continue
            L, a = int(p.blk_len[b]), int(p.blk_pos0[b])
            tot += L * (a + 1) + L * (L - 1) // 2
        return tot
    assert p2.pairs == closed(p2) == 4_409_344
    w4 = synth.workload(4)
    p4, _ = oplan.plan_forest(w4.forest)
    assert (p4.n_tot, p4.n_chunks) == (32768, 4)
    assert p4.pairs == closed(p4) == 520_101_888
    assert max(p4.blk_depth) == 8
    w3 = synth.workload(3)
    p3, _ = oplan.plan_forest(w3.forest)
    assert p3.n_fwd == 8192 and p3.n_res == 0 and max(p3.blk_depth) <= 8
    assert p3.pairs == closed(p3)


def test_identical_prompts_share_one_block_and_readout():
    w3 = synth.workload(3)
    p3, _ = oplan.plan_forest(w3.forest)
    dups = w3.notes["duplicates"]
    assert len(dups) > 0
    for dup, orig in dups.items():
        assert p3.block_map[dup] == p3.block_map[orig]
        assert p3.blk_slot[p3.block_map[dup]] >= 0
    # 256 copies of the template become one resident block with 512 leaves
    w5 = synth.workload(5)
    p5, q5 = oplan.plan_forest(w5.forest, leaf1=w5.leaf1, leaf2=w5.leaf2)
    assert p5.n_res == 32 and p5.n_slots == 512
    assert p5.n_fwd == int(w5.forest.length.sum()) - 256 * 32
    assert len(set(p5.block_map[w5.leaf1 - 1])) == 1


def test_merged_subtrees_pool_children():
    # two identical documents under one template: their questions end up under one block
    par = [-1, 0, 0, 1, 2]
    ln = [4, 6, 6, 3, 3]
    key = np.array([0, 5, 5, 0, 0], np.uint64)
    p, _ = oplan.make_plan(par, ln, key, [0] * 5)
    assert p.n_blocks == 4 and p.n_tot == 16
    assert p.block_map[1] == p.block_map[2]
    assert p.blk_parent[p.block_map[3]] == p.blk_parent[p.block_map[4]] == p.block_map[1]


def test_limits_and_bad_trees():
    def code(par, ln, res=None, **kw):
        res = [0] * len(par) if res is None else res
        with pytest.raises(oplan.PlanError) as e:
            oplan.make_plan(par, ln, np.zeros(len(par), np.uint64), res, **kw)
        return e.value.code
    chain9 = [-1] + list(range(8))
    assert code(chain9, [1] * 9) == oplan.ERR_DEPTH
    oplan.make_plan(chain9[:8], [1] * 8, np.zeros(8, np.uint64), [0] * 8)   # depth 8 is fine
    assert code([-1], [32769]) == oplan.ERR_ROW_TOO_LONG
    oplan.make_plan([-1], [32768], np.zeros(1, np.uint64), [0])
    assert code([-1, 2, 1], [1, 1, 1]) == oplan.ERR_BAD_TREE          # cycle
    assert code([-1, 5], [1, 1]) == oplan.ERR_BAD_TREE                 # orphan
    assert code([-1, 0], [1, 0]) == oplan.ERR_BAD_TREE                 # empty block
    assert code([-1, -1], [4, 4], res=[0, 1]) == oplan.ERR_INVALID_ARG  # resident after forward
    assert code([-1], [4], res=[1]) == oplan.ERR_INVALID_ARG           # nothing to compute
    assert code([-1], [4], max_fwd=100) == oplan.ERR_UNSUPPORTED


def test_chunks_cover_the_forward_tokens():
    w4 = synth.workload(4)
    p4, _ = oplan.plan_forest(w4.forest)
    assert list(p4.chunk_q0) == [0, 8192, 16384, 24576]
    assert list(p4.chunk_q1) == [8192, 16384, 24576, 32768]
    for c in range(4):
        ts = p4.qt_order[p4.chunk_t0[c]:p4.chunk_t1[c]]
        assert sorted(ts) == list(range(p4.chunk_t0[c], p4.chunk_t1[c]))
        work = p4.qt_ent1[ts] - p4.qt_ent0[ts]
        assert np.all(np.diff(work) <= 0)
