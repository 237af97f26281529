"""Pins for the oracle's tree attention (CPU only).

The path-materialising oracle is checked against masked softmax attention over
the packed row (mask from parent links), against the library's causal
attention on chains, and against the invariants the page states: a prompt's
result does not depend on the other prompts packed with it.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import plan as oplan


def _rand_qkv(p, hq, hkv, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((p.n_fwd, hq, d)).astype(np.float16)
    k = rng.standard_normal((p.n_tot, hkv, d)).astype(np.float16)
    v = rng.standard_normal((p.n_tot, hkv, d)).astype(np.float16)
    return q, k, v


@pytest.mark.parametrize("seed", range(10))
def test_paths_match_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    f = synth.random_forest(rng, n_roots=int(rng.integers(1, 3)), max_blocks=int(rng.integers(3, 12)),
                            max_len=int(rng.integers(1, 20)), resident_root=bool(seed % 2))
    try:
        p, _ = oplan.plan_forest(f)
    except oplan.PlanError:
        return
    hq, hkv = [(2, 2), (4, 2), (4, 1)][seed % 3]
    q, k, v = _rand_qkv(p, hq, hkv, 16, seed)
    a = oatt.attend_paths(p, q, k, v, check_shared=True)
    b = oatt.brute_force(p, q, k, v)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    rows = np.arange(p.n_fwd)
    np.testing.assert_allclose(oatt.attend_rows(p, q, k, v, rows), b, rtol=0, atol=1e-12)


def test_chain_is_library_causal_attention():
    # one prompt split over four blocks = plain causal attention over its tokens
    p, _ = oplan.make_plan([-1, 0, 1, 2], [7, 5, 1, 9], np.zeros(4, np.uint64), [0] * 4)
    q, k, v = _rand_qkv(p, 4, 2, 32, 7)
    ours = oatt.attend_paths(p, q, k, v)
    qt = torch.tensor(q.astype(np.float64)).permute(1, 0, 2)
    kt = torch.tensor(k.astype(np.float64)).repeat_interleave(2, dim=1).permute(1, 0, 2)
    vt = torch.tensor(v.astype(np.float64)).repeat_interleave(2, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    np.testing.assert_allclose(ours, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_resident_prefix_is_attended_but_not_computed():
    p, _ = oplan.make_plan([-1, 0], [6, 4], np.zeros(2, np.uint64), [1, 0])
    assert p.n_res == 6 and p.n_fwd == 4
    q, k, v = _rand_qkv(p, 2, 1, 16, 8)
    ours = oatt.attend_paths(p, q, k, v)
    # as one causal sequence of 10 tokens whose first 6 queries are not asked for
    qfull = np.concatenate([np.zeros((6, 2, 16), np.float16), q])
    qt = torch.tensor(qfull.astype(np.float64)).permute(1, 0, 2)
    kt = torch.tensor(k.astype(np.float64)).repeat_interleave(2, dim=1).permute(1, 0, 2)
    vt = torch.tensor(v.astype(np.float64)).repeat_interleave(2, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
    np.testing.assert_allclose(ours, ref.permute(1, 0, 2).numpy()[6:], rtol=0, atol=1e-12)


def test_identical_siblings_do_not_see_each_other():
    # two unmerged option blocks with identical content under one question
    p, _ = oplan.make_plan([-1, 0, 0], [8, 5, 5], np.zeros(3, np.uint64), [0, 0, 0])
    q, k, v = _rand_qkv(p, 2, 2, 16, 9)
    s1, s2 = p.blk_start[1], p.blk_start[2]
    q[s2:s2 + 5] = q[s1:s1 + 5]
    k[s2:s2 + 5] = k[s1:s1 + 5]
    v[s2:s2 + 5] = v[s1:s1 + 5]
    o = oatt.attend_paths(p, q, k, v)
    assert np.array_equal(o[s1:s1 + 5], o[s2:s2 + 5])


def test_result_does_not_depend_on_batch_neighbours():
    # a prompt alone vs the same prompt packed after another row and among siblings
    rng = np.random.default_rng(10)
    d, hq, hkv = 16, 2, 1
    alone, _ = oplan.make_plan([-1, 0, 1], [6, 3, 4], np.zeros(3, np.uint64), [0] * 3)
    qa, ka, va = _rand_qkv(alone, hq, hkv, d, 11)
    oa = oatt.attend_paths(alone, qa, ka, va)
    # packed: another row first, then the same prompt with an extra sibling before its leaf
    packed, _ = oplan.make_plan([-1, -1, 1, 2, 2], [5, 6, 3, 7, 4], np.zeros(5, np.uint64), [0] * 5)
    qp, kp, vp = _rand_qkv(packed, hq, hkv, d, 12)
    src = np.concatenate([np.arange(0, 9), np.arange(9, 13)])             # alone tokens
    dst = np.concatenate([np.arange(5, 14), np.arange(21, 25)])           # same tokens, packed
    qp[dst] = qa[src]
    kp[dst] = ka[src]
    vp[dst] = va[src]
    op = oatt.attend_paths(packed, qp, kp, vp)
    np.testing.assert_allclose(op[dst], oa[src], rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", range(4))
def test_sibling_order_does_not_change_any_token(seed):
    # the same tree given with its children in another input order packs in another order; every
    # token, identified by (input block, offset), keeps its Q/K/V and must keep its output
    rng = np.random.default_rng(300 + seed)
    parent = [-1, 0, 0, 0, 1, 1, 2, 3, 3]
    length = [int(x) for x in rng.integers(1, 9, len(parent))]
    # new input index -> old: every sibling group reversed, then random orders
    order = [0, 3, 2, 1, 5, 4, 6, 8, 7] if seed == 0 else [0] + [int(x) + 1 for x in rng.permutation(len(parent) - 1)]
    new_of = {old: new for new, old in enumerate(order)}
    parent2 = [-1 if parent[o] < 0 else new_of[parent[o]] for o in order]
    length2 = [length[o] for o in order]
    pa, _ = oplan.make_plan(parent, length, np.zeros(len(parent), np.uint64), [0] * len(parent))
    pb, _ = oplan.make_plan(parent2, length2, np.zeros(len(parent), np.uint64), [0] * len(parent))
    qa, ka, va = _rand_qkv(pa, 2, 1, 16, 400 + seed)

    def tokens(p, blk):  # packed indices of input block blk's tokens
        start = int(p.blk_start[p.block_map[blk]])
        return np.arange(start, start + int(p.blk_len[p.block_map[blk]]))
    ia = np.concatenate([tokens(pa, o) for o in order])
    ib = np.concatenate([tokens(pb, n) for n in range(len(order))])
    if seed == 0:
        assert not np.array_equal(ia, ib)   # the packed order does change
    qb, kb, vb = (np.empty_like(x) for x in (qa, ka, va))
    qb[ib], kb[ib], vb[ib] = qa[ia], ka[ia], va[ia]
    oa = oatt.attend_paths(pa, qa, ka, va)
    ob = oatt.attend_paths(pb, qb, kb, vb)
    np.testing.assert_allclose(ob[ib], oa[ia], rtol=0, atol=1e-13)


def test_one_token_block_sees_its_ancestors_and_itself():
    p, _ = oplan.make_plan([-1, 0, 0, 2], [5, 4, 3, 1], np.zeros(4, np.uint64), [0] * 4)
    q, k, v = _rand_qkv(p, 1, 1, 8, 13)
    o = oatt.attend_paths(p, q, k, v)
    t = int(p.blk_start[p.block_map[3]])
    keys = np.array([0, 1, 2, 3, 4, 9, 10, 11, t])
    s = k[keys, 0].astype(np.float64) @ q[t, 0].astype(np.float64) / np.sqrt(8)
    w = np.exp(s - s.max())
    w /= w.sum()
    np.testing.assert_allclose(o[t, 0], w @ v[keys, 0].astype(np.float64), rtol=0, atol=1e-13)


def test_sampled_rows_match_paths_on_workload_two():
    w = synth.workload(2)
    p, _ = oplan.plan_forest(w.forest)
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, w.hq, w.hkv, w.d, w.seed)
    q, k, v = q[:, :4], k[:, :1], v[:, :1]      # one kv group keeps the check quick
    rows = np.array([0, 511, 512, 600, 640, 8191])
    a = oatt.attend_paths(p, q, k, v)
    b = oatt.attend_rows(p, q, k, v, rows)
    np.testing.assert_allclose(a[rows], b, rtol=0, atol=1e-12)


def test_lse_rows_is_library_logsumexp_over_the_brute_mask():
    from scipy.special import logsumexp
    rng = np.random.default_rng(14)
    f = synth.random_forest(rng, n_roots=2, max_blocks=9, max_len=7)
    p, _ = oplan.plan_forest(f)
    q, k, v = _rand_qkv(p, 4, 2, 16, 15)
    m = oplan.brute_mask(p)[p.n_res:]
    ours = oatt.lse_rows(p, q, k, np.arange(p.n_fwd))
    for i in range(p.n_fwd):
        keys = np.nonzero(m[i])[0]
        for h in range(4):
            s = k[keys, h // 2].astype(np.float64) @ q[i, h].astype(np.float64) / 4.0
            assert abs(ours[i, h] - logsumexp(s)) < 1e-12
