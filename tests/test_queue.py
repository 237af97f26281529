"""Request planner: the oracle against the page's numbers and closed forms, the
C-ABI queue (include/tree_queue.h) against the oracle.  CPU only."""
import json
import os

import numpy as np
import pytest

import prefix_tree_packed_gb300 as lib
from oracle import queue as oq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "token_counts.json")


def six_prompts(g, qbase=10):
    """The page's example: template -> state -> question -> option order, 3 questions x 2 orders."""
    prompts = []
    for q in range(g["questions"]):
        for o in range(g["orders"]):
            prompts.append([(1, g["template"]), (2, g["state"]), (qbase + q, g["question"]),
                            (1000 + 10 * q + o + 100 * qbase, g["option"])])
    return prompts, [(2 * q, 2 * q + 1) for q in range(g["questions"])]


# ---------------------------------------------------------------- oracle pins

def test_oracle_cost_worked_example():
    g = json.load(open(GOLDEN))
    prompts, _ = six_prompts(g)
    per_prompt = g["template"] + g["state"] + g["question"] + g["option"]
    assert per_prompt == g["prompt_tokens_printed"]
    separate = g["prompts_printed"] * per_prompt
    tree = oq.request_cost(prompts, resident_keys=[1])
    assert round(separate / tree, 1) == g["reduction_printed"]
    # closed form: state once, each question once, each option order once
    assert tree == g["state"] + g["questions"] * (g["question"] + g["orders"] * g["option"])
    assert oq.request_cost(prompts) == tree + g["template"]


def test_oracle_cost_special_cases():
    # one prompt: its length; identical prompts: counted once; key-0 blocks never shared
    assert oq.request_cost([[(5, 7), (6, 3)]]) == 10
    assert oq.request_cost([[(5, 7), (6, 3)], [(5, 7), (6, 3)]]) == 10
    assert oq.request_cost([[(0, 7)], [(0, 7)]]) == 14
    assert oq.request_cost([[(5, 7), (0, 3)], [(5, 7), (0, 3)]]) == 13
    # same key, different length: different blocks
    assert oq.request_cost([[(5, 7)], [(5, 8)]]) == 15
    # same block under different parents: not shared
    assert oq.request_cost([[(1, 4), (9, 2)], [(2, 4), (9, 2)]]) == 12


def test_oracle_hrrn_crossover():
    # long request (cost L, arrival 0) vs short (cost S, arrival a): 1 + t / (L m) against
    # 1 + (t - a) / (S m); the short one's priority grows faster and overtakes at
    # t* = a L / (L - S): before it the long one goes first, after it the short one
    L, S, a, m = 3000, 300, 50.0, 0.01
    t_star = a * L / (L - S)
    for t, first in ((t_star - 1.0, 1), (t_star + 1.0, 2)):
        q = oq.Queue(long_tokens=0, max_batch_tokens=L, ms_per_token=m)
        q.push(1, 0.0, [[(11, L)]])
        q.push(2, a, [[(12, S)]])
        assert q.pop(t)[1][0] == first
    # equal priorities: the earlier arrival
    assert oq.priority(100, 0.0, 10.0, 0.1) == pytest.approx(2.0)


def test_oracle_fifo_lanes_and_fill():
    q = oq.Queue(fifo=True, long_tokens=8192, max_batch_tokens=8192)
    q.push(1, 0.0, [[(21, 5000)]])
    q.push(2, 1.0, [[(22, 4000)]])
    q.push(3, 2.0, [[(23, 3000)]])
    q.push(4, 3.0, [[(24, 100)]])
    q.push(5, 4.0, [[(25, 9000)]])   # long lane
    assert q.pop(10.0) == (0, [1, 3, 4], 8100)   # 2 does not fit after 1; 3 and 4 do
    assert q.pop(10.0) == (0, [2], 4000)
    assert q.pop(10.0) == (1, [5], 9000)
    assert q.pop(10.0) is None


def test_oracle_shared_prefix_across_requests():
    # two requests on the same 6000-token document: together they cost it once
    q = oq.Queue(long_tokens=0, max_batch_tokens=8192, fifo=True)
    q.push(1, 0.0, [[(7, 6000), (70, 1000)]])
    q.push(2, 0.0, [[(7, 6000), (71, 1000)]])
    assert q.pop(0.0) == (0, [1, 2], 8000)


# ---------------------------------------------------------------- the library against the oracle

def _forest_prefixes(b: lib.Batch):
    """Distinct root-to-node paths of a batch forest as (key, length) tuples."""
    out = []
    for n in range(len(b.parent)):
        path, x = [], n
        while x >= 0:
            path.append((int(b.key[x]), int(b.length[x])))
            x = int(b.parent[x])
        out.append(tuple(reversed(path)))
    return out


def _path(b: lib.Batch, n: int):
    path = []
    while n >= 0:
        path.append((int(b.key[n]), int(b.length[n])))
        n = int(b.parent[n])
    return list(reversed(path))


def test_queue_worked_example_matches_oracle():
    g = json.load(open(GOLDEN))
    prompts, qs = six_prompts(g)
    q = lib.Queue(resident_keys=[1])
    assert q.push(7, 0.0, prompts, qs) == oq.request_cost(prompts, [1])
    b = q.pop(1.0)
    assert b.lane == 0 and b.request_ids == [7] and b.cost == 300
    assert b.resident[0] == 1 and b.parent[0] == -1 and int(b.resident.sum()) == 1
    # every question's readout blocks end the prompts it names
    for i, (a, c) in enumerate(qs):
        assert _path(b, int(b.leaf1[i])) == prompts[a]
        assert _path(b, int(b.leaf2[i])) == prompts[c]
    # the planner takes the batch as it is: forward tokens = cost
    plan = lib.Plan(b.parent, b.length, b.key, b.resident, b.leaf1, b.leaf2)
    assert plan.info.n_tot - plan.info.n_res == b.cost
    assert q.pop(2.0) is None


def _random_request(rng, rid, docs):
    """A request on one of a few shared documents, 1-3 questions x 2 orders, random lengths."""
    doc = int(rng.integers(0, len(docs)))
    prompts, qs = [], []
    for qi in range(int(rng.integers(1, 4))):
        qkey = int(rng.integers(1, 1 << 40))
        qlen = int(rng.integers(8, 200))
        for o in range(2):
            prompts.append([(1, 53), (docs[doc][0], docs[doc][1]), (qkey, qlen),
                            (int(rng.integers(1, 1 << 40)) if rng.random() < 0.9 else 0, int(rng.integers(4, 40)))])
        qs.append((len(prompts) - 2, len(prompts) - 1))
    if rng.random() < 0.2:  # an identical copy of a prompt: shares its readout
        prompts.append(list(prompts[0]))
        qs.append((0, len(prompts) - 1))
    return prompts, qs


@pytest.mark.parametrize("fifo", [False, True])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_queue_matches_oracle_on_random_streams(seed, fifo):
    rng = np.random.default_rng(100 + seed)
    docs = [(int(rng.integers(1 << 41, 1 << 42)), int(rng.integers(100, 5000))) for _ in range(4)]
    opts = lib.queue_default_opts()
    opts.fifo = int(fifo)
    opts.long_tokens = 4096
    q = lib.Queue(opts, resident_keys=[1])
    ref = oq.Queue(fifo=fifo, long_tokens=4096, resident_keys=[1])
    now, rid, popped = 0.0, 0, 0
    reqs = {}
    for step in range(60):
        for _ in range(int(rng.integers(0, 4))):
            prompts, qs = _random_request(rng, rid, docs)
            c = q.push(rid, now, prompts, qs)
            assert c == ref.push(rid, now, prompts, qs)
            reqs[rid] = (prompts, qs)
            rid += 1
        if rid > 0 and rng.random() < 0.1:
            victim = int(rng.integers(0, rid))
            queued = {r.id for r in ref.reqs}
            if victim in queued:
                q.cancel(victim)
                ref.cancel(victim)
            else:
                with pytest.raises(lib.TreeError):
                    q.cancel(victim)
        now += float(rng.uniform(0.0, 40.0))
        if rng.random() < 0.6:
            b = q.pop(now)
            r = ref.pop(now)
            if r is None:
                assert b is None
                continue
            popped += 1
            assert (b.lane, b.request_ids, b.cost) == r
            if b.lane == 0:
                assert b.cost <= 8192 or len(b.request_ids) == 1
            # the forest holds exactly the distinct prefixes of the batch's prompts
            uniq_free = []
            for i in b.request_ids:
                for p in reqs[i][0]:
                    for k in range(1, len(p) + 1):
                        if all(key != 0 for key, _ in p[:k]):
                            uniq_free.append(tuple(p[:k]))
            fp = _forest_prefixes(b)
            assert set(uniq_free) <= set(fp)
            assert len(fp) == len(set(x for x in fp if all(k != 0 for k, _ in x))) + \
                sum(1 for x in fp if any(k == 0 for k, _ in x))
            # questions in request order, each naming its prompts' last blocks
            for j, i in enumerate(b.request_ids):
                prompts, qs = reqs[i]
                for t, (a, c2) in enumerate(qs):
                    n = int(b.request_q0[j]) + t
                    assert _path(b, int(b.leaf1[n])) == [tuple(x) for x in prompts[a]]
                    assert _path(b, int(b.leaf2[n])) == [tuple(x) for x in prompts[c2]]
            plan = lib.Plan(b.parent, b.length, b.key, b.resident, b.leaf1, b.leaf2)
            assert plan.info.n_tot - plan.info.n_res == b.cost
    assert popped > 10
    assert q.info() == (sum(1 for r in ref.reqs if not ref._long(r)), sum(1 for r in ref.reqs if ref._long(r)))


def test_queue_long_lane_and_disable():
    q = lib.Queue()
    assert q.push(1, 0.0, [[(5, 5000)]]) == 5000
    assert q.push(2, 1.0, [[(6, 100)]]) == 100
    assert q.info() == (1, 1)
    b = q.pop(1e6)   # short batches first, however long the long request waited
    assert b.lane == 0 and b.request_ids == [2]
    b = q.pop(1e6)
    assert b.lane == 1 and b.request_ids == [1] and b.cost == 5000
    opts = lib.queue_default_opts()
    opts.long_tokens = 0  # no long lane
    q = lib.Queue(opts)
    q.push(1, 0.0, [[(5, 5000)]])
    assert q.info() == (1, 0)


def test_queue_rejects_bad_requests():
    q = lib.Queue()
    q.push(1, 0.0, [[(5, 10)]])
    cases = [
        (dict(rid=1, prompts=[[(6, 10)]]), lib.TREE_ERR_INVALID_ARG),                    # duplicate id
        (dict(rid=2, prompts=[[(6, 10)]], questions=[(0, 1)]), lib.TREE_ERR_INVALID_ARG),  # no prompt 1
        (dict(rid=3, prompts=[[(6, 0)]]), lib.TREE_ERR_BAD_TREE),                         # empty block
        (dict(rid=4, prompts=[[(i + 1, 2) for i in range(9)]]), lib.TREE_ERR_DEPTH),       # 9 blocks
        (dict(rid=5, prompts=[[(6, 20000), (7, 20000)]]), lib.TREE_ERR_ROW_TOO_LONG),     # prompt > 32768
        (dict(rid=6, prompts=[[(6, 10)], [(6, 10), (7, 3)]], questions=[(0, 1)]),
         lib.TREE_ERR_INVALID_ARG),                                                       # readout prompt is a prefix
        (dict(rid=7, prompts=[]), lib.TREE_ERR_INVALID_ARG),
    ]
    for kw, code in cases:
        with pytest.raises(lib.TreeError) as e:
            q.push(kw["rid"], 0.0, kw["prompts"], kw.get("questions", ()))
        assert e.value.code == code, kw
    assert q.info() == (1, 0)
    with pytest.raises(lib.TreeError):
        q.cancel(99)


def test_queue_keeps_readouts_leaves_and_one_resident_root():
    opts = lib.queue_default_opts()
    opts.fifo = 1
    q = lib.Queue(opts, resident_keys=[1, 2])
    q.push(1, 0.0, [[(9, 10)]], [(0, 0)])
    q.push(2, 1.0, [[(9, 10), (10, 5)]])          # would make request 1's readout block inner
    q.push(3, 2.0, [[(1, 50), (11, 5)]])          # resident root 1
    q.push(4, 3.0, [[(2, 50), (12, 5)]])          # a second resident root: not in the same batch
    b = q.pop(5.0)
    assert b.request_ids == [1, 3]
    b = q.pop(5.0)
    assert b.request_ids == [2, 4]
    assert int(b.resident.sum()) == 1 and b.resident[0] == 1
