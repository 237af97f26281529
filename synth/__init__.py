"""Seeded synthetic workloads for packed prefix-tree attention and letter readout.

This module only draws inputs: block forests (parent / length / content key /
resident flag), question lists, and the random Q/K/V and letter-logit arrays.
It contains none of the method's arithmetic (no packing, masking, RoPE,
attention or decision math), so the CPU oracle and the CUDA path can both take
their inputs from here without sharing any computation.

The five workloads follow the shapes the basal-rs Architecture page describes
("01 / Request path: Batch and prefix tree" and "03 / Packing: Shared state
computed once"): a template block, a document ("state"), question blocks and two
option-order leaves per question, rows of up to 32,768 tokens, trees of depth at
most 8, forwards of up to 8192 tokens.

Random draws use ``numpy.random.default_rng(seed)``; the default seed of a
workload is its number (1..5).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Forest",
    "Workload",
    "workload",
    "WORKLOAD_NAMES",
    "draw_qkv",
    "draw_logits",
    "draw_layer",
    "draw_head",
    "draw_readout_batch",
    "random_forest",
]

WORKLOAD_NAMES = {
    1: "tiny-tree-96tok-h4-d64",
    2: "llama1b-8rows-8192tok-h32kv8-d64",
    3: "llama8b-mixed-8192tok-h32kv8-d128",
    4: "long-row-32768tok-4chunks-h32kv8-d128",
    5: "many-small-256rows-h32kv8-d128",
}


@dataclass
class Forest:
    """Input block forest, one entry per input block (before any merging).

    parent[b]   : index of the parent block, -1 for a root
    length[b]   : tokens in block b (> 0)
    key[b]      : content key; 0 = unique content, equal non-zero keys with
                  equal lengths under the same parent mean identical content
    resident[b] : 1 if the block's K/V already sit in the cache (computed
                  earlier, e.g. the template computed once at startup)
    """

    parent: np.ndarray
    length: np.ndarray
    key: np.ndarray
    resident: np.ndarray

    @property
    def n_blocks(self) -> int:
        return int(self.parent.shape[0])


@dataclass
class Workload:
    number: int
    name: str
    forest: Forest
    hq: int
    hkv: int
    d: int
    theta: float
    seed: int
    # questions: order-1 leaf block, order-2 leaf block, letters, temperature
    leaf1: np.ndarray | None = None
    leaf2: np.ndarray | None = None
    n_letters: np.ndarray | None = None
    temperature: np.ndarray | None = None
    logit_sigma: float = 2.0
    letter_stride: int = 0
    max_fwd: int = 8192
    notes: dict = field(default_factory=dict)


class _Builder:
    def __init__(self):
        self.parent, self.length, self.key, self.resident = [], [], [], []

    def add(self, parent, length, key=0, resident=0):
        self.parent.append(parent)
        self.length.append(length)
        self.key.append(key)
        self.resident.append(resident)
        return len(self.parent) - 1

    def forest(self) -> Forest:
        return Forest(
            parent=np.asarray(self.parent, dtype=np.int32),
            length=np.asarray(self.length, dtype=np.int32),
            key=np.asarray(self.key, dtype=np.uint64),
            resident=np.asarray(self.resident, dtype=np.uint8),
        )


def _w1(seed):
    b = _Builder()
    root = b.add(-1, 64)
    l1 = b.add(root, 16)
    l2 = b.add(root, 16)
    return Workload(
        1, WORKLOAD_NAMES[1], b.forest(), hq=4, hkv=4, d=64, theta=500000.0, seed=seed,
        leaf1=np.array([l1], np.int32), leaf2=np.array([l2], np.int32),
        n_letters=np.array([3], np.int32), temperature=np.array([1.0], np.float32),
        logit_sigma=2.0, letter_stride=3,
    )


def _w2(seed):
    rng = np.random.default_rng(seed)
    b = _Builder()
    tmpl = b.add(-1, 128, key=1, resident=1)
    l1, l2 = [], []
    for _row in range(8):
        doc = b.add(tmpl, 512)
        for _q in range(4):
            qb = b.add(doc, 48)
            l1.append(b.add(qb, 40))
            l2.append(b.add(qb, 40))
    nq = len(l1)
    n = rng.integers(4, 7, size=nq).astype(np.int32)
    temps = np.array([0.7, 1.0, 1.3], np.float32)[rng.integers(0, 3, size=nq)]
    return Workload(
        2, WORKLOAD_NAMES[2], b.forest(), hq=32, hkv=8, d=64, theta=500000.0, seed=seed,
        leaf1=np.array(l1, np.int32), leaf2=np.array(l2, np.int32), n_letters=n,
        temperature=temps.astype(np.float32), logit_sigma=2.0, letter_stride=6,
    )


def _mixed_rows(rng, b: _Builder, total: int, key_counter: list):
    """Rows of random trees until exactly `total` tokens are placed."""
    rem = total
    while rem > 0:
        budget = min(rem, int(rng.integers(2048, 4097)))
        if rem - budget < 16:
            budget = rem
        depth_cap = int(rng.integers(2, 9))
        key_counter[0] += 1
        root_len = min(int(rng.integers(16, 1025)), budget)
        if budget - root_len < 16:
            root_len = budget
        root = b.add(-1, root_len, key=key_counter[0])
        used = root_len
        last = root
        frontier = [(root, 1)]
        while frontier and used < budget:
            blk, dep = frontier.pop(0)
            if dep >= depth_cap:
                continue
            fan = int(rng.integers(1, 7))
            for _ in range(fan):
                if used >= budget:
                    break
                ln = min(int(rng.integers(16, 1025)), budget - used)
                if budget - used - ln < 16:
                    ln = budget - used
                key_counter[0] += 1
                child = b.add(blk, ln, key=key_counter[0])
                used += ln
                last = child
                frontier.append((child, dep + 1))
        if used < budget:
            b.length[last] += budget - used
        rem -= budget


def _w3(seed):
    rng = np.random.default_rng(seed)
    b = _Builder()
    counter = [0]
    _mixed_rows(rng, b, 8192, counter)
    # ~10% of leaves get an identical sibling (same parent, length and key)
    nb = len(b.parent)
    has_child = np.zeros(nb, bool)
    for p in b.parent:
        if p >= 0:
            has_child[p] = True
    leaves = [i for i in range(nb) if not has_child[i]]
    dup_of = {}
    for lf in leaves:
        if rng.random() < 0.1:
            dup_of[b.add(b.parent[lf], b.length[lf], key=b.key[lf])] = lf
    return Workload(
        3, WORKLOAD_NAMES[3], b.forest(), hq=32, hkv=8, d=128, theta=500000.0, seed=seed,
        notes={"duplicates": dup_of},
    )


def _w4(seed):
    b = _Builder()
    doc = b.add(-1, 24576)
    for _ in range(2):
        p = b.add(doc, 2560)
        for ln in (512, 256, 256, 256, 128):
            p = b.add(p, ln)
        b.add(p, 64)
        b.add(p, 64)
    return Workload(
        4, WORKLOAD_NAMES[4], b.forest(), hq=32, hkv=8, d=128, theta=500000.0, seed=seed,
        max_fwd=8192,
    )


def _w5(seed):
    rng = np.random.default_rng(seed)
    b = _Builder()
    l1, l2 = [], []
    for _row in range(256):
        # every row names the same template; the planner keeps one copy
        t = b.add(-1, 32, key=7, resident=1)
        l1.append(b.add(t, int(rng.integers(8, 25))))
        l2.append(b.add(t, int(rng.integers(8, 25))))
    return Workload(
        5, WORKLOAD_NAMES[5], b.forest(), hq=32, hkv=8, d=128, theta=500000.0, seed=seed,
        leaf1=np.array(l1, np.int32), leaf2=np.array(l2, np.int32),
        n_letters=np.full(len(l1), 2, np.int32),
        temperature=np.ones(len(l1), np.float32), logit_sigma=3.0, letter_stride=10,
    )


_BUILDERS = {1: _w1, 2: _w2, 3: _w3, 4: _w4, 5: _w5}


def workload(number: int, seed: int | None = None) -> Workload:
    """The block forest and shapes of workload `number` (1..5)."""
    return _BUILDERS[number](number if seed is None else seed)


def draw_qkv(n_fwd: int, n_tot: int, hq: int, hkv: int, d: int, seed: int):
    """Q for the forward tokens, K/V for every token of the KV space; f16 ~ N(0,1).

    Rows of K for resident tokens are taken as already rotated (their RoPE was
    applied when they were computed); rows of forward tokens are pre-RoPE.
    """
    rng = np.random.default_rng(seed + 1000)
    q = rng.standard_normal((n_fwd, hq, d), dtype=np.float32).astype(np.float16)
    k = rng.standard_normal((n_tot, hkv, d), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((n_tot, hkv, d), dtype=np.float32).astype(np.float16)
    return q, k, v


def draw_layer(n_fwd: int, n_res: int, hidden: int, hq: int, hkv: int, d: int, ffn: int, seed: int):
    """Random-init weights of one Llama layer and its inputs, all f16.

    Linear weights ~ N(0, 1/fan_in) (rows = outputs), norm weights ~ 1 + N(0, 0.1^2);
    hidden states of the forward tokens ~ N(0,1); the resident tokens' (already
    rotated) keys and values ~ N(0,1).  There are no trained weights: the shapes
    are those of the model, the values random.
    """
    rng = np.random.default_rng(seed + 4000)

    def lin(n_out, n_in):
        return (rng.standard_normal((n_out, n_in), dtype=np.float32) / np.sqrt(n_in)).astype(np.float16)

    w = {
        "w_in": (1.0 + 0.1 * rng.standard_normal(hidden)).astype(np.float16),
        "wq": lin(hq * d, hidden), "wk": lin(hkv * d, hidden), "wv": lin(hkv * d, hidden),
        "wo": lin(hidden, hq * d),
        "w_post": (1.0 + 0.1 * rng.standard_normal(hidden)).astype(np.float16),
        "wgu": lin(2 * ffn, hidden), "wd": lin(hidden, ffn),
    }
    w["wqkv"] = np.concatenate([w["wq"], w["wk"], w["wv"]])  # the fused projection's layout
    x = rng.standard_normal((n_fwd, hidden), dtype=np.float32).astype(np.float16)
    res_k = rng.standard_normal((n_res, hkv * d), dtype=np.float32).astype(np.float16)
    res_v = rng.standard_normal((n_res, hkv * d), dtype=np.float32).astype(np.float16)
    return w, x, res_k, res_v


def draw_head(hidden: int, stride: int, seed: int):
    """The final RMSNorm weight and the LM-head rows of the answer letters (f16, random init)."""
    rng = np.random.default_rng(seed + 5000)
    w_final = (1.0 + 0.1 * rng.standard_normal(hidden)).astype(np.float16)
    w_letters = (rng.standard_normal((stride, hidden), dtype=np.float32) / np.sqrt(hidden)).astype(np.float16)
    return w_final, w_letters


def draw_logits(n_slots: int, stride: int, sigma: float, seed: int):
    rng = np.random.default_rng(seed + 2000)
    return (rng.standard_normal((n_slots, stride)) * sigma).astype(np.float32)


def draw_readout_batch(n_questions: int = 65536, seed: int = 5):
    """Standalone readout batch: 2..10 letters, logits ~ N(0,3), T in {0.5,1,2}.

    Question q reads logits rows 2q (order 1) and 2q+1 (order 2) of a
    (2*n_questions, 10) f32 buffer.
    """
    rng = np.random.default_rng(seed + 3000)
    stride = 10
    logits = (rng.standard_normal((2 * n_questions, stride)) * 3.0).astype(np.float32)
    n = rng.integers(2, 11, size=n_questions).astype(np.int32)
    temps = np.array([0.5, 1.0, 2.0], np.float32)[rng.integers(0, 3, size=n_questions)]
    r1 = (2 * np.arange(n_questions)).astype(np.int32)
    r2 = (2 * np.arange(n_questions) + 1).astype(np.int32)
    return dict(logits=logits, stride=stride, r1=r1, r2=r2, n_letters=n, temperature=temps)


def random_forest(rng, n_roots: int = 2, max_blocks: int = 12, max_len: int = 9,
                  dup_prob: float = 0.2, resident_root: bool = False) -> Forest:
    """Small random forest for brute-force checks (tiny blocks, shallow trees).

    Block ids are shuffled so that parents do not always precede children, and
    some siblings are given identical (length, key) so that they merge.
    """
    b = _Builder()
    nodes = []
    for r in range(n_roots):
        res = 1 if (resident_root and r == 0) else 0
        nodes.append((b.add(-1, int(rng.integers(1, max_len + 1)), key=0, resident=res), 1))
    while len(b.parent) < max_blocks:
        p, dep = nodes[int(rng.integers(0, len(nodes)))]
        if dep >= 8:
            continue
        if rng.random() < dup_prob:
            ln = 3
            key = 99
        else:
            ln = int(rng.integers(1, max_len + 1))
            key = 0
        nodes.append((b.add(p, ln, key=key), dep + 1))
    f = b.forest()
    if resident_root:
        # keep the resident root first so that resident tokens lead the packing
        perm = np.concatenate([[0], 1 + rng.permutation(f.n_blocks - 1)])
    else:
        perm = rng.permutation(f.n_blocks)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(f.n_blocks)
    parent = np.where(f.parent[perm] >= 0, inv[np.maximum(f.parent[perm], 0)], -1).astype(np.int32)
    return Forest(parent=parent, length=f.length[perm].copy(), key=f.key[perm].copy(),
                  resident=f.resident[perm].copy())
